// CUDA kernels (sm_103a) of the mixed-format paged decode-attention library.
//
// Method: "Minima-KV: Retention-Preserving KV Cache Compression with
// Mixed-Format Paged Attention" (arXiv 2608.23834), abstract on the
// mlsanity.com paper page: Recent/Anchor pages in FP8, Stale pages in packed
// TQ3, format-specific kernels producing partial attention states, and a
// globally normalised online-softmax merge with no dense shadow.  Formats and
// layouts are defined in include/mkv.h ("Storage formats").
//
// Kernels:
//   mkv_append_kernel  -- FP8 quantise new K/V rows into their pages
//   mkv_demote_kernel  -- FP8 page -> TQ3 page (dequantise, rotate, RMS scale,
//                         Lloyd-Max codes, pack)
//   mkv_qprep_kernel   -- per (request, kv head): q rows (and q' = R q) as
//                         fp16 hi/lo MMA fragments
//   mkv_decode_kernel  -- persistent, warp-specialised partial-attention
//                         kernel over both formats
//   mkv_merge_kernel   -- LSE merge: TQ3 partials in the rotated domain,
//                         one R^T, then FP8 partials; writes out and lse
#include "mkv_internal.h"

#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <mutex>

namespace mkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz: bound on any wait
constexpr float kLazyRescale = 8.0f;               // log2 units a max may grow before O is rescaled
constexpr float kFp8PScale = 512.0f;               // keeps p * s in fp16 normal range for FP8 V

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// two E4M3 codes (low byte -> low half) to an f16x2 register; exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ bool sign_neg(const uint64_t (&signs)[4], int i) {
  // select the word instead of indexing the parameter array (keeps it out of local memory)
  const int w = i >> 6;
  const uint64_t word = w == 0 ? signs[0] : w == 1 ? signs[1] : w == 2 ? signs[2] : signs[3];
  return (word >> (i & 63)) & 1ull;
}

// TQ3: four 3-bit codes held as nibbles in sel[15:0] -> two f16x2 registers
// (codes 0,1) and (codes 2,3).  PRMT looks the low and the high byte of each
// level up in 8-byte tables, then interleaves them.
__device__ __forceinline__ void tq3_lookup4(uint32_t sel, const Lut& t, uint32_t& h01, uint32_t& h23) {
  const uint32_t lo = __byte_perm(t.lo_a, t.lo_b, sel);
  const uint32_t hi = __byte_perm(t.hi_a, t.hi_b, sel);
  h01 = __byte_perm(lo, hi, 0x5140);
  h23 = __byte_perm(lo, hi, 0x7362);
}
// One 12-byte unit (32 codes) -> eight nibble selectors (4 codes each).
__device__ __forceinline__ void tq3_unit_selectors(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t (&s)[8]) {
  const uint32_t m0 = w0 & 0x77777777u, m1 = w1 & 0x77777777u, m2 = w2 & 0x77777777u;
  const uint32_t e = ((w0 >> 3) & 0x11111111u) | ((w1 >> 2) & 0x22222222u) | ((w2 >> 1) & 0x44444444u);
  s[0] = m0; s[1] = m0 >> 16; s[2] = m1; s[3] = m1 >> 16;
  s[4] = m2; s[5] = m2 >> 16; s[6] = e;  s[7] = e >> 16;
}

// ============================================================== append
// FP8-quantise one row (one token, kv head, K|V) into its page: the calling
// warp holds the row; s = fp16(amax / 448), codes = e4m3_rn_satfinite(x / s)
// with IEEE fp32 divisions.
__device__ __forceinline__ void fp8_append_row(const void* src_rows, size_t row, int bf16, uint8_t* plane, int P,
                                               int kv, int pos, int lane) {
  float x[8];
  if (bf16) {
    const uint4 raw = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src_rows) + row)[lane];
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(b2[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else {
    const float4* f4 = reinterpret_cast<const float4*>(static_cast<const float*>(src_rows) + row) + 2 * lane;
    const float4 a = f4[0], b = f4[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
  const __half s16 = __float2half_rn(__fdiv_rn(amax, 448.0f));
  const float s = __half2float(s16);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint16_t two = 0;
    if (s != 0.f) {
      const float a = __fdiv_rn(x[2 * i], s), b = __fdiv_rn(x[2 * i + 1], s);
      // cvt packs its first source into the upper byte
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(b), "f"(a));
    }
    c[i] = two;
  }
  if (kv == 0) {
    uint2 w;
    w.x = c[0] | (c[1] << 16);
    w.y = c[2] | (c[3] << 16);
    *reinterpret_cast<uint2*>(plane + pos * kHeadDim + 8 * lane) = w;
  } else {
    uint8_t* base = plane + (pos >> 1) * (2 * kHeadDim) + (pos & 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      base[2 * (8 * lane + 2 * i)] = static_cast<uint8_t>(c[i] & 0xff);
      base[2 * (8 * lane + 2 * i + 1)] = static_cast<uint8_t>(c[i] >> 8);
    }
  }
  if (lane == 0) reinterpret_cast<__half*>(plane + P * kHeadDim)[pos] = s16;
}

// One warp per (token, kv head, K|V) row.
__global__ void __launch_bounds__(256) mkv_append_kernel(AppendParams p) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int nrows = p.ntok * p.Hkv * 2;
  if (warp >= nrows) return;
  const int kv = warp & 1;
  const int h = (warp >> 1) % p.Hkv;
  const int tok = (warp >> 1) / p.Hkv;
  const uint32_t dst = p.dest[tok];
  const int slot = static_cast<int>(dst >> 8), pos = static_cast<int>(dst & 0xff);
  const int P = p.P;
  uint8_t* plane = p.fp8_layer + static_cast<int64_t>(slot) * p.fp8_page_bytes +
                   static_cast<int64_t>(h) * 2 * (P * (kHeadDim + 2)) + kv * (P * (kHeadDim + 2));
  fp8_append_row(kv ? p.v : p.k, (static_cast<size_t>(tok) * p.Hkv + h) * kHeadDim, p.kv_bf16, plane, P, kv, pos,
                 lane);
}

// ============================================================== demote
// One block per (page pair, layer, kv head, K|V plane).  Each warp encodes
// rows (dequantise, sign flip, 8-stage FWHT, RMS scale, threshold count);
// the block then packs 12-byte units and writes the TQ3 plane.
__global__ void __launch_bounds__(256) mkv_demote_kernel(DemoteParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const int P = p.P;
  uint8_t* codes = dsm;                                                 // [P][256]
  __half* sig = reinterpret_cast<__half*>(dsm + P * kHeadDim);          // [P]
  int job = blockIdx.x;
  const int kv = job & 1;
  job >>= 1;
  const int h = job % p.Hkv;
  job /= p.Hkv;
  const int layer = job % p.L;
  const int pair = job / p.L;
  const int2 sl = p.pairs[pair];
  const int fp8_plane = P * (kHeadDim + 2);
  const int tq3_plane = P * (3 * kHeadDim / 8 + 2);
  const uint8_t* src = p.fp8_arena + layer * p.fp8_layer_stride + static_cast<int64_t>(sl.x) * p.fp8_page_bytes +
                       static_cast<int64_t>(h) * 2 * fp8_plane + kv * fp8_plane;
  uint8_t* dst = p.tq3_arena + layer * p.tq3_layer_stride + static_cast<int64_t>(sl.y) * p.tq3_page_bytes +
                 static_cast<int64_t>(h) * 2 * tq3_plane + kv * tq3_plane;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __half* sc = reinterpret_cast<const __half*>(src + P * kHeadDim);
  for (int t = warp; t < P; t += 8) {
    uint8_t b[8];
    if (kv == 0) {
      const uint2 w = *reinterpret_cast<const uint2*>(src + t * kHeadDim + 8 * lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        b[i] = (w.x >> (8 * i)) & 0xff;
        b[4 + i] = (w.y >> (8 * i)) & 0xff;
      }
    } else {
      const uint8_t* r = src + (t >> 1) * (2 * kHeadDim) + (t & 1);
#pragma unroll
      for (int i = 0; i < 8; ++i) b[i] = r[2 * (8 * lane + i)];
    }
    const float s = __half2float(sc[t]);
    float x[8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t f2 = e4m3x2_to_f16x2(b[2 * i] | (b[2 * i + 1] << 8));
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f2));
      x[2 * i] = f.x * s;
      x[2 * i + 1] = f.y * s;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
    const __half sg16 = __float2half_rn(__fsqrt_rn(ss * (1.0f / kHeadDim)));
    const float sg = __half2float(sg16);
    // y = H (signs .* x) / 16; element index j = 8*lane + i
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (sign_neg(p.signs, 8 * lane + i)) x[i] = -x[i];
#pragma unroll
    for (int hs = 1; hs < 8; hs <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if ((i & hs) == 0) {
          const float a = x[i], c = x[i + hs];
          x[i] = a + c;
          x[i + hs] = a - c;
        }
      }
    }
#pragma unroll
    for (int lm = 1; lm < 32; lm <<= 1) {
      const bool upper = (lane & lm) != 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = __shfl_xor_sync(kFull, x[i], lm);
        x[i] = upper ? (o - x[i]) : (x[i] + o);
      }
    }
    uint8_t cd[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y = x[i] * (1.0f / 16.0f);
      const float u = (sg != 0.f) ? __fdiv_rn(y, sg) : 0.f;
      int k = 0;
#pragma unroll
      for (int q = 0; q < 7; ++q) k += (p.thr[q] <= u) ? 1 : 0;
      cd[i] = static_cast<uint8_t>(k);
    }
    uint2 packed;
    packed.x = cd[0] | (cd[1] << 8) | (cd[2] << 16) | (cd[3] << 24);
    packed.y = cd[4] | (cd[5] << 8) | (cd[6] << 16) | (cd[7] << 24);
    *reinterpret_cast<uint2*>(codes + t * kHeadDim + 8 * lane) = packed;
    if (lane == 0) sig[t] = sg16;
  }
  __syncthreads();
  // pack units: word w -> unit w/3, word index k = w%3
  const int nwords = P * (kHeadDim / 32) * 3;
  uint32_t* out = reinterpret_cast<uint32_t*>(dst);
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) {
    const int unit = w / 3, k = w - 3 * (w / 3);
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int e0 = 8 * k + i, e1 = 24 + i;
      uint32_t c0, c1;
      if (kv == 0) {
        const int t = unit / (kHeadDim / 32), j0 = (unit % (kHeadDim / 32)) * 32;
        c0 = codes[t * kHeadDim + j0 + e0];
        c1 = codes[t * kHeadDim + j0 + e1];
      } else {
        const int v = unit / (kHeadDim / 16), j0 = (unit % (kHeadDim / 16)) * 16;
        c0 = codes[(2 * v + (e0 & 1)) * kHeadDim + j0 + (e0 >> 1)];
        c1 = codes[(2 * v + (e1 & 1)) * kHeadDim + j0 + (e1 >> 1)];
      }
      word |= (c0 & 7u) << (4 * i);
      word |= ((c1 >> k) & 1u) << (4 * i + 3);
    }
    out[w] = word;
  }
  __half* osc = reinterpret_cast<__half*>(dst + P * (3 * kHeadDim / 8));
  for (int t = threadIdx.x; t < P; t += blockDim.x) osc[t] = sig[t];
}

// ============================================================== dequantise (export)
// One warp per (token, kv head, K|V) row of the requested pages: FP8 rows are
// e4m3 * s; TQ3 rows are unpacked from their 12-byte units, scaled by the
// stored levels and sigma, and rotated back (H, then the signs, then 1/16).
__global__ void __launch_bounds__(256) mkv_dequant_kernel(DequantParams p) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int P = p.P;
  const int nrows = p.npages * P * p.Hkv * 2;
  if (warp >= nrows) return;
  const int kv = warp & 1;
  const int h = (warp >> 1) % p.Hkv;
  const int t_all = (warp >> 1) / p.Hkv;          // token index in the output
  const int pg = t_all / P, t = t_all % P;
  const int2 pe = p.pages[pg];
  const int tier = pe.y >> 16, nvalid = pe.y & 0xffff;
  float x[8];
  if (t >= nvalid) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.f;
  } else if (tier != 3) {
    const int plane = P * (kHeadDim + 2);
    const uint8_t* base = p.fp8_layer + static_cast<int64_t>(pe.x) * p.fp8_page_bytes +
                          static_cast<int64_t>(h) * 2 * plane + kv * plane;
    const float s = __half2float(reinterpret_cast<const __half*>(base + P * kHeadDim)[t]);
    uint8_t b[8];
    if (kv == 0) {
      const uint2 w = *reinterpret_cast<const uint2*>(base + t * kHeadDim + 8 * lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        b[i] = (w.x >> (8 * i)) & 0xff;
        b[4 + i] = (w.y >> (8 * i)) & 0xff;
      }
    } else {
      const uint8_t* r = base + (t >> 1) * (2 * kHeadDim) + (t & 1);
#pragma unroll
      for (int i = 0; i < 8; ++i) b[i] = r[2 * (8 * lane + i)];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t f2 = e4m3x2_to_f16x2(b[2 * i] | (b[2 * i + 1] << 8));
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f2));
      x[2 * i] = f.x * s;
      x[2 * i + 1] = f.y * s;
    }
  } else {
    const int plane = P * (3 * kHeadDim / 8 + 2);
    const uint8_t* base = p.tq3_layer + static_cast<int64_t>(pe.x) * p.tq3_page_bytes +
                          static_cast<int64_t>(h) * 2 * plane + kv * plane;
    const float sg = __half2float(reinterpret_cast<const __half*>(base + P * (3 * kHeadDim / 8))[t]);
    // lane holds dims 8*lane .. 8*lane+7
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = 8 * lane + i;
      int unit, e;
      if (kv == 0) {
        unit = t * (kHeadDim / 32) + j / 32;
        e = j % 32;
      } else {
        unit = (t >> 1) * (kHeadDim / 16) + j / 16;
        e = 2 * (j % 16) + (t & 1);
      }
      const uint32_t* w = reinterpret_cast<const uint32_t*>(base + 12 * unit);
      int code;
      if (e < 24) {
        code = (w[e >> 3] >> (4 * (e & 7))) & 7;
      } else {
        const int i2 = e - 24;
        code = ((w[0] >> (4 * i2 + 3)) & 1) | (((w[1] >> (4 * i2 + 3)) & 1) << 1) | (((w[2] >> (4 * i2 + 3)) & 1) << 2);
      }
      x[i] = sg * p.level[code];
    }
    // x <- H x (natural order), then signs and 1/16
#pragma unroll
    for (int hs = 1; hs < 8; hs <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if ((i & hs) == 0) {
          const float a = x[i], c = x[i + hs];
          x[i] = a + c;
          x[i + hs] = a - c;
        }
    }
#pragma unroll
    for (int lm = 1; lm < 32; lm <<= 1) {
      const bool upper = (lane & lm) != 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = __shfl_xor_sync(kFull, x[i], lm);
        x[i] = upper ? (o - x[i]) : (x[i] + o);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[i] *= (1.0f / 16.0f);
      if (sign_neg(p.signs, 8 * lane + i)) x[i] = -x[i];
    }
  }
  const size_t off = (static_cast<size_t>(t_all) * p.Hkv + h) * kHeadDim + 8 * lane;
  void* dst = kv ? p.v_out : p.k_out;
  if (p.out_bf16) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(dst) + off;
    uint4 pk;
    __nv_bfloat162 q0 = __floats2bfloat162_rn(x[0], x[1]), q1 = __floats2bfloat162_rn(x[2], x[3]);
    __nv_bfloat162 q2 = __floats2bfloat162_rn(x[4], x[5]), q3 = __floats2bfloat162_rn(x[6], x[7]);
    pk.x = *reinterpret_cast<uint32_t*>(&q0);
    pk.y = *reinterpret_cast<uint32_t*>(&q1);
    pk.z = *reinterpret_cast<uint32_t*>(&q2);
    pk.w = *reinterpret_cast<uint32_t*>(&q3);
    *reinterpret_cast<uint4*>(o) = pk;
  } else {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(dst) + off);
    o[0] = make_float4(x[0], x[1], x[2], x[3]);
    o[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
}

// ============================================================== q prep
// Per (request, kv head): the QK warps' MMA A fragments of the group's query
// rows for both formats -- FP8 pages score against q, TQ3 pages against
// q' = R q (signs, then H, then 1/16).  Rows 0-7 of the A tile hold fp16(q_h)
// of heads h = 0..G-1, rows 8-15 the fp16 residual q_h - fp16(q_h), so the
// two halves of the S accumulator add up to an fp32-accurate score.
// Fragment layout: [(b*Hkv + kvh)*2 + fmt][lane 32][k-step 16][4 regs], with
// lane (g, c) = (lane/4, lane%4) covering dims 64c + 4j .. 64c + 4j + 3.
__global__ void __launch_bounds__(320) mkv_qprep_kernel(QprepParams p) {
  __shared__ __align__(16) float qs[2][kMaxGroup][kHeadDim];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x / p.Hkv, kvh = blockIdx.x % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kMaxGroup) {
    // fused single-token append: warp 8 writes the K row, warp 9 the V row
    if (p.append) {
      const int kv = warp - kMaxGroup;
      const uint32_t dst = p.dest[b];
      const int slot = static_cast<int>(dst >> 8), pos = static_cast<int>(dst & 0xff);
      uint8_t* plane = p.fp8_layer + static_cast<int64_t>(slot) * p.fp8_page_bytes +
                       static_cast<int64_t>(kvh) * 2 * (p.P * (kHeadDim + 2)) + kv * (p.P * (kHeadDim + 2));
      fp8_append_row(kv ? p.v : p.k, (static_cast<size_t>(b) * p.Hkv + kvh) * kHeadDim, p.kv_bf16, plane, p.P, kv,
                     pos, lane);
    }
    __syncthreads();
    return;
  }
  float x[8];
  if (warp < p.G) {
    const size_t off = (static_cast<size_t>(b) * p.Hq + kvh * p.G + warp) * kHeadDim + 8 * lane;
    if (p.q_bf16) {
      const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + off);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b2[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
    } else {
      const float4* f4 = reinterpret_cast<const float4*>(static_cast<const float*>(p.q) + off);
      const float4 a = f4[0], c = f4[1];
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) qs[0][warp][8 * lane + i] = x[i];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (sign_neg(p.signs, 8 * lane + i)) x[i] = -x[i];
#pragma unroll
  for (int hs = 1; hs < 8; hs <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & hs) == 0) {
        const float a = x[i], c = x[i + hs];
        x[i] = a + c;
        x[i + hs] = a - c;
      }
  }
#pragma unroll
  for (int lm = 1; lm < 32; lm <<= 1) {
    const bool upper = (lane & lm) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(kFull, x[i], lm);
      x[i] = upper ? (o - x[i]) : (x[i] + o);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) qs[1][warp][8 * lane + i] = x[i] * (1.0f / 16.0f);
  __syncthreads();
  if (threadIdx.x >= 256) return;
  const int fmt = threadIdx.x >> 7, L = (threadIdx.x >> 2) & 31, j0 = 4 * (threadIdx.x & 3);
  const int g = L >> 2, c = L & 3;
  uint4* dst = reinterpret_cast<uint4*>(p.qfrag + ((static_cast<size_t>(b) * p.Hkv + kvh) * 2 + fmt) * 2048 +
                                        L * 64 + 4 * j0);
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const float4 v = *reinterpret_cast<const float4*>(&qs[fmt][g][64 * c + 4 * (j0 + jj)]);
    const float vv[4] = {v.x, v.y, v.z, v.w};
    float hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      hi[i] = __half2float(__float2half_rn(vv[i]));
      lo[i] = vv[i] - hi[i];
    }
    dst[jj] = make_uint4(pack_half2(hi[0], hi[1]), pack_half2(lo[0], lo[1]), pack_half2(hi[2], hi[3]),
                         pack_half2(lo[2], lo[3]));
  }
}

// ============================================================== decode
// Persistent, warp-specialised partial-attention kernel; one CTA per SM.
//   warps 0-7   QK warps: S = Q K^T on mma.sync m16n8k16 (A = q rows from the
//               q-prep fragments, B = K dequantised in registers), online
//               softmax in log2 units with a lazy rescale, P (scaled by the V
//               row scales, fp16) handed to the partner PV warp.
//   warps 8-15  PV warps: O^T += V^T P^T (A = V dequantised in registers).
// Page blocks move by cp.async.bulk copies (K codes, K scales, V codes, V
// scales of each page) into a ring of kNumStages shared-memory slots whose
// mbarriers count the bytes.  A TQ3 block is 128 tokens (8 tiles of 16: pair
// i takes tile i); an FP8 block is 64 tokens (4 tiles: pair i takes tile i%4
// of the blocks with parity i/4, and FP8 pieces are padded to an even number
// of blocks so every pair sees the last one).  There is no producer warp:
// thread 0 issues the first kNumStages blocks and afterwards the last warp to
// release a slot (found with a shared-memory counter) issues the block
// kNumStages further on into it.
// The host cut the launch's global sequence of blocks into one contiguous,
// cost-balanced piece list per CTA; each (CTA, group) piece ends with the 8
// pairs' states merged into one partial state (m, l, o) per q head.
constexpr int kPairs = 8;
constexpr int kDecWarps = 2 * kPairs;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kNumStages = 5;
constexpr int kFp8Tokens = 64;            // tokens per FP8 block
constexpr int kTq3Tokens = 128;           // tokens per TQ3 block
constexpr int kSlotBytes = 2 * (kFp8Tokens * kHeadDim + 2 * kFp8Tokens);   // an FP8 block; a TQ3 block fits
constexpr uint32_t kWaitHintNs = 20000;   // try_wait suspend hint

template <int FMT>
struct Blk {                               // a block of format FMT in a slot
  static constexpr int kTokens = FMT == 0 ? kFp8Tokens : kTq3Tokens;
  static constexpr int kRow = FMT == 0 ? kHeadDim : 3 * kHeadDim / 8;      // K row bytes
  static constexpr int kCode = kTokens * kRow;
  static constexpr int kK = 0, kKs = kCode, kV = kCode + 2 * kTokens, kVs = 2 * kCode + 2 * kTokens;
  static constexpr int kBytes = 2 * (kCode + 2 * kTokens);
};
static_assert(Blk<1>::kBytes <= kSlotBytes, "a TQ3 block must fit a slot");

struct PSlot {                                   // P handoff QK warp -> PV warp
  uint2 pb[32];                                  // B fragments (fp16 P' pairs) per lane
  float alpha[kMaxGroup];                        // O rescale factor per head
  int32_t rescale;
  int32_t pad[7];
};

struct DecSmem {
  uint8_t* ring;
  PSlot* pslot;                                  // [kPairs][2]
  float* acc;                                    // [4][kMaxGroup][D]: pair sums of a piece's O
  float* epi_m;                                  // [kPairs][kMaxGroup]
  float* epi_l;
  uint64_t* full;                                // [kNumStages]
  uint64_t* pfull;                               // [kPairs][2]
  uint64_t* pempty;                              // [kPairs][2]
  int* release;                                  // [kNumStages] warps done with the slot
  int* issued;                                   // blocks issued so far (for the abort drain)
  int* abort_flag;
};
constexpr int kDecSmemRing = kNumStages * kSlotBytes;
constexpr int kDecSmemP = kPairs * 2 * static_cast<int>(sizeof(PSlot));
constexpr int kDecSmemEpi = 4 * kMaxGroup * kHeadDim * 4 + 2 * kPairs * kMaxGroup * 4;
constexpr int kDecSmemBars = (kNumStages + 4 * kPairs) * 8 + (kNumStages + 2) * 4 + 8;
constexpr int kDecSmemBytes = kDecSmemRing + kDecSmemP + kDecSmemEpi + kDecSmemBars;

__device__ __forceinline__ DecSmem dec_carve(uint8_t* base) {
  DecSmem s;
  s.ring = base;
  s.pslot = reinterpret_cast<PSlot*>(base + kDecSmemRing);
  s.acc = reinterpret_cast<float*>(base + kDecSmemRing + kDecSmemP);
  s.epi_m = s.acc + 4 * kMaxGroup * kHeadDim;
  s.epi_l = s.epi_m + kPairs * kMaxGroup;
  s.full = reinterpret_cast<uint64_t*>(s.epi_l + kPairs * kMaxGroup);
  s.pfull = s.full + kNumStages;
  s.pempty = s.pfull + 2 * kPairs;
  s.release = reinterpret_cast<int*>(s.pempty + 2 * kPairs);
  s.issued = s.release + kNumStages;
  s.abort_flag = s.issued + 1;
  return s;
}

__device__ __forceinline__ bool aborted(const DecSmem& sm) {
  return *reinterpret_cast<volatile int*>(sm.abort_flag) != 0;
}
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kWaitHintNs)
      : "memory");
  return ok != 0;
}
// Bounded wait (kWaitCycles) that also gives up once any warp of the CTA has
// aborted; the thread sleeps in try_wait until the phase completes.
__device__ __forceinline__ bool dec_wait(const DecSmem& sm, uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait_hint(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity)) return true;
    if (aborted(sm)) return false;
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(err, kErrWaitTimeout);
      *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
      return false;
    }
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One CTA's piece list: piece si covers global blocks [pstart, pstart + ptotal).
// Holds only the fields the loops use.
struct PieceCursor {
  int si, s1;
  int pstart, ptotal;
  int entry, blk, nstages, part;   // from the Segment
  int fmt, b, kvh, gend;           // from the Group (gend: one past its last entry)
  __device__ void load(const DecodeParams& p) {
    const Segment* sp = p.segs + si;
    const int grp = sp->group;
    entry = sp->entry;
    blk = sp->blk;
    nstages = sp->nstages;
    part = sp->part;
    const Group* gp = p.groups + grp;
    fmt = gp->fmt;
    b = gp->b;
    kvh = gp->kvh;
    gend = gp->entry0 + gp->nentry;
    ptotal = fmt ? nstages : nstages + (nstages & 1);
  }
  __device__ bool start(const DecodeParams& p, int s0, int s1_) {
    si = s0;
    s1 = s1_;
    pstart = 0;
    if (si >= s1) return false;
    load(p);
    return true;
  }
  __device__ bool next_piece(const DecodeParams& p) {
    pstart += ptotal;
    if (++si >= s1) return false;
    load(p);
    return true;
  }
  __device__ bool seek(const DecodeParams& p, int gi) {
    while (gi >= pstart + ptotal)
      if (!next_piece(p)) return false;
    return true;
  }
  // Block k of the piece: first page entry, block within that page (FP8 at
  // P = 128 has two blocks per page), pages (TQ3 at P = 64 has two pages per
  // block), and valid tokens (0 for an FP8 padding block).
  __device__ int block(const DecodeParams& p, int k, int& e, int& half, int& npages) const {
    if (k >= nstages) return 0;
    if (fmt == 0) {
      const int bpp = p.P / kFp8Tokens;                // blocks per page: 1 or 2
      const int bb = blk + k;
      e = entry + bb / bpp;
      half = bb % bpp;
      npages = 1;
      return min(kFp8Tokens, p.entries[e].nvalid - kFp8Tokens * half);
    }
    const int ppb = kTq3Tokens / p.P;                  // pages per block: 2 or 1
    e = entry + k * ppb;
    half = 0;
    npages = min(ppb, gend - e);
    return npages * p.P;
  }
  // valid tokens of block k only (consumers)
  __device__ int tokens(const DecodeParams& p, int k) const {
    if (k >= nstages) return 0;
    if (fmt == 0) {
      const int bpp = p.P / kFp8Tokens;
      const int bb = blk + k;
      return min(kFp8Tokens, p.entries[entry + bb / bpp].nvalid - kFp8Tokens * (bb % bpp));
    }
    const int ppb = kTq3Tokens / p.P;
    return min(ppb, gend - (entry + k * ppb)) * p.P;
  }
};

// Issue global block gi (cursor positioned on its piece) into its slot: four
// bulk copies per page, or a plain arrive for a padding block.  False on a
// bad plan.
__device__ __noinline__ bool dec_issue(const DecodeParams& p, const DecSmem& sm, const PieceCursor& cur, int gi) {
  const int slot = gi % kNumStages;
  atomicMax(sm.issued, gi + 1);
  int e = 0, half = 0, npages = 0;
  if (cur.block(p, gi - cur.pstart, e, half, npages) <= 0) {
    mbar_arrive(&sm.full[slot]);   // padding block: the phase completes without bytes
    return true;
  }
  const int fmt = cur.fmt;
  const int nslots = fmt ? p.tq3_slots : p.fp8_slots;
  const int row = fmt ? 3 * kHeadDim / 8 : kHeadDim;
  const int plane = p.P * (row + 2);
  const int btok = fmt ? kTq3Tokens : kFp8Tokens;          // tokens per block in the slot layout
  const int ptok = fmt ? p.P : kFp8Tokens;                 // tokens copied per page
  for (int i = 0; i < npages; ++i) {
    const PageEntry pe = p.entries[e + i];
    // a request's last page may still be receiving its new token from the
    // preceding (q-prep + append) kernel: copy it only after that kernel is done
    if (pe.tail) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (pe.slot < 0 || pe.slot >= nslots) {
      atomicOr(p.err, kErrBadPlan);
      *reinterpret_cast<volatile int*>(sm.abort_flag) = 1;
      mbar_arrive(&sm.full[slot]);
      return false;
    }
  }
  uint8_t* st = sm.ring + slot * kSlotBytes;
  const uint32_t code = ptok * row;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(&sm.full[slot], npages * 2 * (code + 2 * ptok));
  for (int i = 0; i < npages; ++i) {
    const PageEntry pe = p.entries[e + i];
    const uint8_t* hp = (fmt ? p.tq3_layer : p.fp8_layer) +
                        static_cast<int64_t>(pe.slot) * (fmt ? p.tq3_page_bytes : p.fp8_page_bytes) +
                        static_cast<int64_t>(cur.kvh) * 2 * plane;
    const int tok0 = ptok * half;                          // first token of the copy within its page
    const int t = ptok * i;                                // first token of the copy within the block
    bulk_g2s(st + t * row, hp + tok0 * row, code, &sm.full[slot]);
    bulk_g2s(st + btok * row + 2 * t, hp + p.P * row + 2 * tok0, 2 * ptok, &sm.full[slot]);
    bulk_g2s(st + btok * row + 2 * btok + t * row, hp + plane + tok0 * row, code, &sm.full[slot]);
    bulk_g2s(st + 2 * btok * row + 2 * btok + 2 * t, hp + plane + p.P * row + 2 * tok0, 2 * ptok,
             &sm.full[slot]);
  }
  return true;
}

// Issue block gi + kNumStages if it exists (cursor positioned at or before it).
__device__ __noinline__ void dec_issue_ahead(const DecodeParams& p, const DecSmem& sm, PieceCursor cur, int gi) {
  if (cur.seek(p, gi + kNumStages)) dec_issue(p, sm, cur, gi + kNumStages);
}

// A warp is done with block gi's slot (`users` warps use a block of this
// format).  The last one to say so issues block gi + kNumStages into the slot.
__device__ __forceinline__ void dec_release(const DecodeParams& p, const DecSmem& sm, int gi, int users,
                                            const PieceCursor& cur) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    __threadfence_block();
    const int slot = gi % kNumStages;
    if (atomicAdd(&sm.release[slot], 1) == users - 1) {
      sm.release[slot] = 0;
      __threadfence_block();
      if (!aborted(sm)) dec_issue_ahead(p, sm, cur, gi);
    }
  }
}

// S for one 16-token tile (two n8 halves, tokens g and 8+g of the tile as B
// columns); FP8 K rows are row-major, the thread's 64 dims are 64 bytes.
__device__ __forceinline__ void dec_qk_fp8(const uint8_t* kt, int g, int c, const uint32_t (&qa)[16][4],
                                           float (&s0)[4], float (&s1)[4]) {
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint4 w0 = *reinterpret_cast<const uint4*>(kt + g * kHeadDim + 64 * c + 16 * q4);
    const uint4 w1 = *reinterpret_cast<const uint4*>(kt + (8 + g) * kHeadDim + 64 * c + 16 * q4);
    const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w};
    const uint32_t x1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 4 * q4 + i;
      mma16816(s0, qa[j][0], qa[j][1], qa[j][2], qa[j][3], e4m3x2_to_f16x2(x0[i]), e4m3x2_to_f16x2(x0[i] >> 16));
      mma16816(s1, qa[j][0], qa[j][1], qa[j][2], qa[j][3], e4m3x2_to_f16x2(x1[i]), e4m3x2_to_f16x2(x1[i] >> 16));
    }
  }
}

// S for one 16-token tile of TQ3 K: row (8u + g) units 2c, 2c+1 (24 bytes at 24c).
__device__ __forceinline__ void dec_qk_tq3(const uint8_t* kt, int g, int c, const uint32_t (&qa)[16][4],
                                           const Lut& lut, float (&s0)[4], float (&s1)[4]) {
  const uint8_t* r0 = kt + g * 96 + 24 * c;
  const uint8_t* r1 = kt + (8 + g) * 96 + 24 * c;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint2 a01 = *reinterpret_cast<const uint2*>(r0 + 12 * half);
    const uint32_t a2 = *reinterpret_cast<const uint32_t*>(r0 + 12 * half + 8);
    const uint2 b01 = *reinterpret_cast<const uint2*>(r1 + 12 * half);
    const uint32_t b2 = *reinterpret_cast<const uint32_t*>(r1 + 12 * half + 8);
    uint32_t sa[8], sb[8];
    tq3_unit_selectors(a01.x, a01.y, a2, sa);
    tq3_unit_selectors(b01.x, b01.y, b2, sb);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int j = 8 * half + s;
      uint32_t x0, x1, y0, y1;
      tq3_lookup4(sa[s], lut, x0, x1);
      tq3_lookup4(sb[s], lut, y0, y1);
      mma16816(s0, qa[j][0], qa[j][1], qa[j][2], qa[j][3], x0, x1);
      mma16816(s1, qa[j][0], qa[j][1], qa[j][2], qa[j][3], y0, y1);
    }
  }
}

// O^T += V^T P^T for FP8 V: pair-rows c and c+4 of the tile, dims [32g, 32g+32)
__device__ __forceinline__ void dec_pv_fp8(const uint8_t* vt, int g, int c, uint2 pb, float (&o)[16][4]) {
  const uint8_t* ra = vt + c * (2 * kHeadDim) + 64 * g;
  const uint8_t* rb = vt + (c + 4) * (2 * kHeadDim) + 64 * g;
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint4 wa = *reinterpret_cast<const uint4*>(ra + 16 * q4);
    const uint4 wb = *reinterpret_cast<const uint4*>(rb + 16 * q4);
    const uint32_t xa[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t xb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      mma16816(o[4 * q4 + i], e4m3x2_to_f16x2(xa[i]), e4m3x2_to_f16x2(xa[i] >> 16), e4m3x2_to_f16x2(xb[i]),
               e4m3x2_to_f16x2(xb[i] >> 16), pb.x, pb.y);
  }
}

// O^T += V^T P^T for TQ3 V: pair-rows c and c+4, units 2g, 2g+1 (24 bytes at 24g)
__device__ __forceinline__ void dec_pv_tq3(const uint8_t* vt, int g, int c, uint2 pb, const Lut& lut,
                                           float (&o)[16][4]) {
  const uint8_t* ra = vt + c * 192 + 24 * g;
  const uint8_t* rb = vt + (c + 4) * 192 + 24 * g;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint2 a01 = *reinterpret_cast<const uint2*>(ra + 12 * half);
    const uint32_t a2 = *reinterpret_cast<const uint32_t*>(ra + 12 * half + 8);
    const uint2 b01 = *reinterpret_cast<const uint2*>(rb + 12 * half);
    const uint32_t b2 = *reinterpret_cast<const uint32_t*>(rb + 12 * half + 8);
    uint32_t sa[8], sb[8];
    tq3_unit_selectors(a01.x, a01.y, a2, sa);
    tq3_unit_selectors(b01.x, b01.y, b2, sb);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t x0, x1, y0, y1;
      tq3_lookup4(sa[s], lut, x0, x1);
      tq3_lookup4(sb[s], lut, y0, y1);
      mma16816(o[8 * half + s], x0, x1, y0, y1, pb.x, pb.y);
    }
  }
}

// The piece's partial state.  QK warps have published (m, l) per pair and
// head; PV warps have left O rescaled to the common max in four buffers
// (pair i + pair i+4 in buffer i).  Every thread writes its share, summing the
// buffers in a fixed order so the result does not depend on timing.
__device__ __forceinline__ void dec_piece_write(const DecodeParams& p, const DecSmem& sm, int part, int G) {
  const int t = threadIdx.x, d = t & 255;
  float* dst = p.part + static_cast<size_t>(part) * G * (2 + kHeadDim);
  for (int h = t >> 8; h < G; h += 2) {
    const float* a = sm.acc + h * kHeadDim + d;
    constexpr int kBuf = kMaxGroup * kHeadDim;
    dst[h * (2 + kHeadDim) + 2 + d] = (a[0] + a[kBuf]) + (a[2 * kBuf] + a[3 * kBuf]);
    if (d == 0) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kPairs; ++w) M = fmaxf(M, sm.epi_m[w * kMaxGroup + h]);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kPairs; ++w) {
          const float mw = sm.epi_m[w * kMaxGroup + h];
          if (mw != -INFINITY) L += ex2(mw - M) * sm.epi_l[w * kMaxGroup + h];
        }
      }
      dst[h * (2 + kHeadDim)] = M;
      dst[h * (2 + kHeadDim) + 1] = L;
    }
  }
}

__device__ void dec_qk_warp(const DecodeParams& p, const DecSmem& sm, int s0, int s1) {
  const int pair = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const Lut lut = p.lut;
  const float scale = p.score_scale;
  const int G = p.G;
  uint32_t qa[16][4];
  int pj = 0;
  bool dep_waited = false;
  PieceCursor cur;
  for (bool more = cur.start(p, s0, s1); more; more = cur.next_piece(p)) {
    const int fmt = cur.fmt;
    if (!dep_waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      dep_waited = true;
    }
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.qfrag + ((static_cast<size_t>(cur.b) * p.Hkv + cur.kvh) * 2 + fmt) * kQfragWords + lane * 64);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint4 v = src[j];
        qa[j][0] = v.x;
        qa[j][1] = v.y;
        qa[j][2] = v.z;
        qa[j][3] = v.w;
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    const int tile = fmt ? pair : (pair & 3);
    const int step = fmt ? 1 : 2;
    const int users = fmt ? 2 * kPairs : kPairs;
    for (int k = fmt ? 0 : (pair >> 2); k < cur.ptotal; k += step) {
      const int gi = cur.pstart + k;
      const int slot = gi % kNumStages;
      const bool ok = dec_wait(sm, &sm.full[slot], (gi / kNumStages) & 1, p.err);
      const int nv = cur.tokens(p, k) - kTileTokens * tile;
      if (ok && nv > 0) {
        const uint8_t* st = sm.ring + slot * kSlotBytes;
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        const __half2* ks;
        const __half2* vs;
        if (fmt == 0) {
          dec_qk_fp8(st + Blk<0>::kK + tile * kTileTokens * kHeadDim, g, c, qa, sa, sb);
          ks = reinterpret_cast<const __half2*>(st + Blk<0>::kKs + tile * kTileTokens * 2);
          vs = reinterpret_cast<const __half2*>(st + Blk<0>::kVs + tile * kTileTokens * 2);
        } else {
          dec_qk_tq3(st + Blk<1>::kK + tile * kTileTokens * 96, g, c, qa, lut, sa, sb);
          ks = reinterpret_cast<const __half2*>(st + Blk<1>::kKs + tile * kTileTokens * 2);
          vs = reinterpret_cast<const __half2*>(st + Blk<1>::kVs + tile * kTileTokens * 2);
        }
        const float2 k01 = __half22float2(ks[c]), k89 = __half22float2(ks[4 + c]);
        const float2 v01 = __half22float2(vs[c]), v89 = __half22float2(vs[4 + c]);
        float sc[4];
        sc[0] = (sa[0] + sa[2]) * (k01.x * scale);
        sc[1] = (sa[1] + sa[3]) * (k01.y * scale);
        sc[2] = (sb[0] + sb[2]) * (k89.x * scale);
        sc[3] = (sb[1] + sb[3]) * (k89.y * scale);
        if (g >= G) {
          sc[0] = sc[1] = sc[2] = sc[3] = -INFINITY;
        } else if (nv < kTileTokens) {
          if (2 * c >= nv) sc[0] = -INFINITY;
          if (2 * c + 1 >= nv) sc[1] = -INFINITY;
          if (8 + 2 * c >= nv) sc[2] = -INFINITY;
          if (9 + 2 * c >= nv) sc[3] = -INFINITY;
        }
        float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
        float alpha = 1.f;
        const bool rescale = __any_sync(kFull, mt > m_run + kLazyRescale);
        if (rescale) {
          const float m_new = fmaxf(m_run, mt);
          alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - m_new);
          m_run = m_new;
          l_run *= alpha;
        }
        // m_run stays -inf only for heads g >= G (all their scores -inf)
        const float mref = (m_run == -INFINITY) ? 0.f : m_run;
        float pr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) pr[i] = (sc[i] == -INFINITY) ? 0.f : ex2(sc[i] - mref);
        l_run += (pr[0] + pr[1]) + (pr[2] + pr[3]);
        // masked tokens give exactly 0 (their scale bytes may be stale)
        const float vsc = fmt == 0 ? kFp8PScale : 1.f;
        const float w0 = pr[0] == 0.f ? 0.f : pr[0] * (v01.x * vsc);
        const float w1 = pr[1] == 0.f ? 0.f : pr[1] * (v01.y * vsc);
        const float w2 = pr[2] == 0.f ? 0.f : pr[2] * (v89.x * vsc);
        const float w3 = pr[3] == 0.f ? 0.f : pr[3] * (v89.y * vsc);
        const uint2 pb = make_uint2(pack_half2(w0, w1), pack_half2(w2, w3));
        const int ps = pj & 1;
        PSlot& slotp = sm.pslot[2 * pair + ps];
        bool okp = true;
        if (pj >= 2) okp = dec_wait(sm, &sm.pempty[2 * pair + ps], ((pj >> 1) - 1) & 1, p.err);
        if (okp) {
          slotp.pb[lane] = pb;
          if (c == 0) slotp.alpha[g] = alpha;
          if (lane == 0) slotp.rescale = rescale ? 1 : 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.pfull[2 * pair + ps]);
        ++pj;
      }
      dec_release(p, sm, gi, users, cur);
    }
    // end of the piece: publish (m, l) of head g, then merge with the PV warps
    float l = l_run;
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (c == 0) {
      sm.epi_m[pair * kMaxGroup + g] = (g < G) ? m_run : -INFINITY;
      sm.epi_l[pair * kMaxGroup + g] = (g < G) ? l : 0.f;
    }
    named_bar(1, kDecThreads);   // (m, l) published
    named_bar(1, kDecThreads);   // pairs 4-7 stored their O
    named_bar(1, kDecThreads);   // pairs 0-3 added theirs
    dec_piece_write(p, sm, cur.part, G);
    named_bar(1, kDecThreads);   // buffers and (m, l) free again
  }
}

__device__ void dec_pv_warp(const DecodeParams& p, const DecSmem& sm, int s0, int s1) {
  const int pair = (threadIdx.x >> 5) - kPairs, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const Lut lut = p.lut;
  const int G = p.G;
  float o[16][4];
  int pj = 0;
  PieceCursor cur;
  for (bool more = cur.start(p, s0, s1); more; more = cur.next_piece(p)) {
    const int fmt = cur.fmt;
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const int tile = fmt ? pair : (pair & 3);
    const int step = fmt ? 1 : 2;
    const int users = fmt ? 2 * kPairs : kPairs;
    for (int k = fmt ? 0 : (pair >> 2); k < cur.ptotal; k += step) {
      const int gi = cur.pstart + k;
      const int slot = gi % kNumStages;
      const bool ok = dec_wait(sm, &sm.full[slot], (gi / kNumStages) & 1, p.err);
      const int nv = cur.tokens(p, k) - kTileTokens * tile;
      if (ok && nv > 0) {
        const int ps = pj & 1;
        const PSlot& slotp = sm.pslot[2 * pair + ps];
        const bool okp = dec_wait(sm, &sm.pfull[2 * pair + ps], (pj >> 1) & 1, p.err);
        const uint2 pb = slotp.pb[lane];
        const int rescale = slotp.rescale;
        float a0 = 1.f, a1 = 1.f;
        if (rescale) {
          a0 = slotp.alpha[2 * c];
          a1 = slotp.alpha[2 * c + 1];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.pempty[2 * pair + ps]);
        ++pj;
        if (okp) {
          if (rescale) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              o[i][0] *= a0;
              o[i][1] *= a1;
              o[i][2] *= a0;
              o[i][3] *= a1;
            }
          }
          const uint8_t* st = sm.ring + slot * kSlotBytes;
          if (fmt == 0)
            dec_pv_fp8(st + Blk<0>::kV + tile * (kTileTokens / 2) * (2 * kHeadDim), g, c, pb, o);
          else
            dec_pv_tq3(st + Blk<1>::kV + tile * (kTileTokens / 2) * 192, g, c, pb, lut, o);
        }
      }
      dec_release(p, sm, gi, users, cur);
    }
    // end of the piece: wait for the QK warps' (m, l), rescale O to the common
    // max of each head, and combine pairs i and i+4 into buffer i (i < 4)
    named_bar(1, kDecThreads);
    const float osc = fmt == 0 ? 1.f / kFp8PScale : 1.f;
    float f0, f1;
    {
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < kPairs; ++w) {
        M0 = fmaxf(M0, sm.epi_m[w * kMaxGroup + 2 * c]);
        M1 = fmaxf(M1, sm.epi_m[w * kMaxGroup + 2 * c + 1]);
      }
      const float m0 = sm.epi_m[pair * kMaxGroup + 2 * c], m1 = sm.epi_m[pair * kMaxGroup + 2 * c + 1];
      f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - M0) * osc;
      f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - M1) * osc;
    }
    float* buf = sm.acc + (pair & 3) * kMaxGroup * kHeadDim;
    if (pair >= 4) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int d = 32 * g + 2 * i;
        if (2 * c < G)
          *reinterpret_cast<float2*>(buf + (2 * c) * kHeadDim + d) = make_float2(o[i][0] * f0, o[i][2] * f0);
        if (2 * c + 1 < G)
          *reinterpret_cast<float2*>(buf + (2 * c + 1) * kHeadDim + d) = make_float2(o[i][1] * f1, o[i][3] * f1);
      }
    }
    named_bar(1, kDecThreads);
    if (pair < 4) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int d = 32 * g + 2 * i;
        if (2 * c < G) {
          float2* q = reinterpret_cast<float2*>(buf + (2 * c) * kHeadDim + d);
          const float2 v = *q;
          *q = make_float2(o[i][0] * f0 + v.x, o[i][2] * f0 + v.y);
        }
        if (2 * c + 1 < G) {
          float2* q = reinterpret_cast<float2*>(buf + (2 * c + 1) * kHeadDim + d);
          const float2 v = *q;
          *q = make_float2(o[i][1] * f1 + v.x, o[i][3] * f1 + v.y);
        }
      }
    }
    named_bar(1, kDecThreads);
    dec_piece_write(p, sm, cur.part, G);
    named_bar(1, kDecThreads);
  }
}

__global__ void __launch_bounds__(kDecThreads, 1) mkv_decode_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DecSmem sm = dec_carve(smem);
  const int s0 = p.cta_seg[blockIdx.x], s1 = p.cta_seg[blockIdx.x + 1];
  // the merge kernel that follows waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumStages; ++i) {
      mbar_init(&sm.full[i], 1);
      sm.release[i] = 0;
    }
    for (int i = 0; i < 2 * kPairs; ++i) {
      mbar_init(&sm.pfull[i], 1);
      mbar_init(&sm.pempty[i], 1);
    }
    *sm.issued = 0;
    *sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the first kNumStages blocks
    PieceCursor cur;
    if (cur.start(p, s0, s1)) {
      for (int gi = 0; gi < kNumStages && cur.seek(p, gi); ++gi)
        if (!dec_issue(p, sm, cur, gi)) break;
    }
  }
  __syncthreads();
  if (s0 < s1) {
    if (threadIdx.x < kPairs * 32)
      dec_qk_warp(p, sm, s0, s1);
    else
      dec_pv_warp(p, sm, s0, s1);
  }
  // every issued block is consumed on the normal path; after an abort, wait
  // (bounded) for copies still in flight before the CTA exits
  __syncthreads();
  if (threadIdx.x == 0 && aborted(sm)) {
    const int n = *sm.issued;
    for (int k = n > kNumStages ? n - kNumStages : 0; k < n; ++k) {
      const long long t0 = clock64();
      while (!mbar_try_wait(&sm.full[k % kNumStages], (k / kNumStages) & 1))
        if (clock64() - t0 > kWaitCycles) break;
    }
  }
}

// ============================================================== merge
// One block (256 threads, thread = dim) per (request, kv head, q head).  The
// partial states' (m, l) are staged in shared memory; the TQ3 partials merge
// in the rotated domain, R^T is applied once (FWHT across the block, then the
// signs and 1/16), the FP8 partials join, and out = O / L,
// lse = (M + log2 L) ln 2.
constexpr int kMergeStage = 256;   // partial states staged per pass

// Merge partial states [first, first + count) of head h at dim d.
__device__ __forceinline__ void merge_range(const float* part, int stride, int h, int first, int count, int d,
                                            float* sm_m, float* sm_l, float& Mout, float& Lout, float& oout) {
  float M = -INFINITY;
  for (int base = 0; base < count; base += kMergeStage) {
    const int cnt = min(kMergeStage, count - base);
    __syncthreads();
    if (d < cnt) {
      const float* pj = part + static_cast<size_t>(first + base + d) * stride + h * (2 + kHeadDim);
      sm_m[d] = pj[0];
      sm_l[d] = pj[1];
    }
    __syncthreads();
    for (int j = 0; j < cnt; ++j) M = fmaxf(M, sm_m[j]);
  }
  float L = 0.f, o = 0.f;
  if (M != -INFINITY) {
    for (int base = 0; base < count; base += kMergeStage) {
      const int cnt = min(kMergeStage, count - base);
      __syncthreads();
      if (d < cnt) {
        const float* pj = part + static_cast<size_t>(first + base + d) * stride + h * (2 + kHeadDim);
        const float mj = pj[0];
        sm_m[d] = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
        sm_l[d] = pj[1];
      }
      __syncthreads();
      const float* col = part + static_cast<size_t>(first + base) * stride + h * (2 + kHeadDim) + 2 + d;
      int j = 0;
      for (; j + 4 <= cnt; j += 4) {
        const float v0 = col[static_cast<size_t>(j) * stride], v1 = col[static_cast<size_t>(j + 1) * stride];
        const float v2 = col[static_cast<size_t>(j + 2) * stride], v3 = col[static_cast<size_t>(j + 3) * stride];
        o += sm_m[j] * v0 + sm_m[j + 1] * v1 + sm_m[j + 2] * v2 + sm_m[j + 3] * v3;
      }
      for (; j < cnt; ++j) o += sm_m[j] * col[static_cast<size_t>(j) * stride];
      for (int jj = 0; jj < cnt; ++jj) L += sm_m[jj] * sm_l[jj];
    }
  }
  Mout = M;
  Lout = L;
  oout = o;
}

__global__ void __launch_bounds__(256) mkv_merge_kernel(MergeParams p) {
  __shared__ float xs[kHeadDim];
  __shared__ float sm_m[kMergeStage], sm_l[kMergeStage];
  // launched as a programmatic dependent of the decode kernel: wait for its
  // partial states before reading them
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int h = blockIdx.x % p.G;
  const int bk = blockIdx.x / p.G;
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  const MergeDesc md = p.desc[bk];
  const int d = threadIdx.x, lane = d & 31;
  const int stride = p.G * (2 + kHeadDim);
  float Ms, Ls, os, Mf, Lf, of;
  merge_range(p.part, stride, h, md.tq3_first, md.tq3_count, d, sm_m, sm_l, Ms, Ls, os);
  // o_S = R^T o'_S = signs .* (H o'_S) / 16: butterflies over lane bits by
  // shuffle, over warp bits through shared memory
#pragma unroll
  for (int lm = 1; lm < 32; lm <<= 1) {
    const float other = __shfl_xor_sync(kFull, os, lm);
    os = (lane & lm) ? (other - os) : (os + other);
  }
  for (int bm = 32; bm < kHeadDim; bm <<= 1) {
    __syncthreads();
    xs[d] = os;
    __syncthreads();
    const float other = xs[d ^ bm];
    os = (d & bm) ? (other - os) : (os + other);
  }
  os *= (1.0f / 16.0f);
  if (sign_neg(p.signs, d)) os = -os;
  merge_range(p.part, stride, h, md.fp8_first, md.fp8_count, d, sm_m, sm_l, Mf, Lf, of);
  const float M = fmaxf(Ms, Mf);
  const float fs = (Ms == -INFINITY) ? 0.f : exp2f(Ms - M);
  const float ff = (Mf == -INFINITY) ? 0.f : exp2f(Mf - M);
  const float L = Ls * fs + Lf * ff;
  const int hq = kvh * p.G + h;
  p.out[(static_cast<size_t>(b) * p.Hq + hq) * kHeadDim + d] = (os * fs + of * ff) / L;
  if (d == 0) p.lse[b * p.Hq + hq] = (M + log2f(L)) * 0.69314718055994530942f;
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  const int rows = p.ntok * p.Hkv * 2;
  const int blocks = (rows + 7) / 8;
  if (blocks > 0) mkv_append_kernel<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_demote(const DemoteParams& p, cudaStream_t s) {
  const int blocks = p.npairs * p.L * p.Hkv * 2;
  const size_t smem = static_cast<size_t>(p.P) * kHeadDim + p.P * 2;
  if (blocks > 0) mkv_demote_kernel<<<blocks, 256, smem, s>>>(p);
  return cudaGetLastError();
}

size_t decode_smem_bytes() { return kDecSmemBytes; }

// Fixed scratch for the allocation-free decode entry point: 8 MiB of partial
// states, compiled into the library so a call never needs to allocate.
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchBytes / sizeof(float)];

cudaError_t noalloc_scratch(float** ptr, size_t* bytes) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static float* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    // host code must not use the symbol itself as a device address: ask the
    // runtime for this device's copy (the current device is `dev`)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(p);
  }
  *ptr = addr[dev];
  *bytes = kNoallocScratchBytes;
  return cudaSuccess;
}
int decode_threads() { return kDecThreads; }

cudaError_t launch_dequant(const DequantParams& p, cudaStream_t s) {
  const int rows = p.npages * p.P * p.Hkv * 2;
  if (rows > 0) mkv_dequant_kernel<<<(rows + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_qprep(const QprepParams& p, cudaStream_t s) {
  if (p.n * p.Hkv > 0) mkv_qprep_kernel<<<p.n * p.Hkv, 320, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(mkv_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.n_ctas <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_ctas);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = kDecSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mkv_decode_kernel, p);
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.n * p.Hkv <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n * p.Hkv * p.G);
  cfg.blockDim = dim3(kHeadDim);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mkv_merge_kernel, p);
}

}  // namespace mkv
