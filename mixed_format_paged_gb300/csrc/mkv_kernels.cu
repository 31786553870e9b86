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
//   mkv_decode_kernel  -- persistent partial-attention kernel over both
//                         formats: 12 independent warps per CTA, each with its
//                         own ring of bulk-copied page blocks (<1>); <2> serves
//                         two query tokens per batch entry (8 warps, several
//                         query tokens per request)
//   mkv_merge_kernel   -- LSE merge: TQ3 partials in the rotated domain,
//                         one R^T, then FP8 partials; writes out and lse
#include "mkv_internal.h"

#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <atomic>

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
// A 1-D bulk copy global -> shared counted by an mbarrier, with an L2 cache
// policy (createpolicy): KV page data is read once per launch and should not
// push the small, reused data (plan tables, q, partial states) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
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
// One 12-byte unit (32 codes) -> eight nibble selectors (4 codes each):
// codes 8k+i sit in nibbles of word k already (mask off bit 3); codes 24+i
// gather bit 3 of nibble i of the three words.  PRMT reads selector bits
// [15:0] only, so the upper four codes of a word take a 16-bit right shift.
__device__ __forceinline__ void tq3_unit_selectors(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t (&s)[8]) {
  const uint32_t m0 = w0 & 0x77777777u, m1 = w1 & 0x77777777u, m2 = w2 & 0x77777777u;
  const uint32_t e = ((w0 >> 3) & 0x11111111u) | ((w1 >> 2) & 0x22222222u) | ((w2 >> 1) & 0x44444444u);
  s[0] = m0; s[1] = m0 >> 16; s[2] = m1; s[3] = m1 >> 16;
  s[4] = m2; s[5] = m2 >> 16; s[6] = e;  s[7] = e >> 16;
}

// ============================================================== append
// FP8-quantise one row (one token, kv head, K|V) held by the calling warp:
// s = fp16(amax / 448), codes = e4m3_rn_satfinite(x / s) with IEEE fp32
// divisions.  Lane l gets the codes of dims 8l .. 8l+7 (two per c[i]).
__device__ __forceinline__ void fp8_quantize_row(const void* src_rows, size_t row, int bf16, int lane,
                                                 uint32_t (&c)[4], __half& s16) {
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
  s16 = __float2half_rn(__fdiv_rn(amax, 448.0f));
  const float s = __half2float(s16);
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
}
// Store a quantised row at position pos of a K (kv = 0) or V (kv = 1) plane
// of P tokens: K codes row-major, V codes pair-interleaved, then P fp16 scales.
// Works on a page plane in global memory and on a staged block in shared
// memory alike (a staged FP8 block has the layout of a 16-token page).
__device__ __forceinline__ void fp8_store_row(uint8_t* plane, int P, int kv, int pos, int lane,
                                              const uint32_t (&c)[4], __half s16) {
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
  uint32_t c[4];
  __half s16;
  fp8_quantize_row(kv ? p.v : p.k, (static_cast<size_t>(tok) * p.Hkv + h) * kHeadDim, p.kv_bf16, lane, c, s16);
  fp8_store_row(plane, P, kv, pos, lane, c, s16);
}

// ============================================================== demote
// One block per (page pair, layer, kv head, K|V plane); each warp encodes
// rows and packs them straight into the TQ3 plane.  Lane l holds dims
// 8l .. 8l + 7 of a row (dequantise, sign flip, 8-stage FWHT, RMS scale,
// threshold count).
//
// One row's codes: nibble i of the result is the code of dim 8 lane + i;
// sg16 gets the row's fp16 sigma.  code = #{k : tau_k <= y / sigma}, decided
// as tau_k * sigma <= y (sigma > 0): the two differ only within about one
// fp32 rounding of a threshold.  sigma == 0 gives u = 0, code 4 (tau_1 ..
// tau_4 <= 0 < tau_5).
__device__ __forceinline__ uint32_t demote_row(float (&x)[8], uint32_t sg8, const float (&thr)[7], int lane,
                                               __half& sg16) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
  sg16 = __float2half_rn(__fsqrt_rn(ss * (1.0f / kHeadDim)));
  const float sg = __half2float(sg16);
  // y = H (signs .* x) / 16; element index j = 8*lane + i
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if ((sg8 >> i) & 1u) x[i] = -x[i];
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
  if (sg == 0.f) return 0x44444444u;
  float tq[7];
#pragma unroll
  for (int q = 0; q < 7; ++q) tq[q] = thr[q] * sg;
  uint32_t nib = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = x[i] * (1.0f / 16.0f);
    uint32_t k = 0;
#pragma unroll
    for (int q = 0; q < 7; ++q) k += (tq[q] <= y) ? 1u : 0u;
    nib |= k << (4 * i);
  }
  return nib;
}
// Eight e4m3 codes (two words, code i in byte i) times the row scale s.
__device__ __forceinline__ void demote_dequant(uint32_t w0, uint32_t w1, float s, float (&x)[8]) {
  const uint32_t w[2] = {w0, w1};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t f2 = e4m3x2_to_f16x2(w[h] >> (16 * i));
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f2));
      x[4 * h + 2 * i] = f.x * s;
      x[4 * h + 2 * i + 1] = f.y * s;
    }
  }
}
// Nibbles 0..3 of a and b interleaved: nibble 2i = a's nibble i, 2i + 1 = b's.
__device__ __forceinline__ uint32_t nibble_zip(uint32_t a, uint32_t b) {
  a &= 0xFFFFu;
  b &= 0xFFFFu;
  a = (a | (a << 8)) & 0x00FF00FFu;
  a = (a | (a << 4)) & 0x0F0F0F0Fu;
  b = (b | (b << 8)) & 0x00FF00FFu;
  b = (b | (b << 4)) & 0x0F0F0F0Fu;
  return a | (b << 4);
}
// A unit's word from the nibble word of its own codes and the nibble word e
// of its codes 24..31 (bit k of each of those goes to bit 3 of nibble i).
__device__ __forceinline__ uint32_t tq3_word(uint32_t nib, uint32_t e, int k) {
  return (nib & 0x77777777u) | (((e >> k) & 0x11111111u) << 3);
}

__global__ void __launch_bounds__(256) mkv_demote_kernel(DemoteParams p) {
  const int P = p.P;
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
  __half* osc = reinterpret_cast<__half*>(dst + P * (3 * kHeadDim / 8));
  // the rotation signs of this lane's dims (select, not index, the parameter array)
  const uint32_t sg8 = static_cast<uint32_t>(
      (lane < 8 ? p.signs[0] : lane < 16 ? p.signs[1] : lane < 24 ? p.signs[2] : p.signs[3]) >> (8 * (lane & 7))) & 0xFFu;
  float thr[7];
#pragma unroll
  for (int q = 0; q < 7; ++q) thr[q] = p.thr[q];
  if (kv == 0) {
    // K: row t's unit l / 4 is lanes 4u .. 4u + 3; lane 4u + k (k < 3) writes
    // word k (its own 8 codes), lane 4u + 3's codes fill the words' bit 3s
    for (int t = warp; t < P; t += 8) {
      const uint2 w = *reinterpret_cast<const uint2*>(src + t * kHeadDim + 8 * lane);
      float x[8];
      demote_dequant(w.x, w.y, __half2float(sc[t]), x);
      __half sg16;
      const uint32_t nib = demote_row(x, sg8, thr, lane, sg16);
      const uint32_t e = __shfl_sync(kFull, nib, lane | 3);
      const int k = lane & 3;
      if (k != 3) reinterpret_cast<uint32_t*>(dst + t * (3 * kHeadDim / 8))[3 * (lane >> 2) + k] = tq3_word(nib, e, k);
      if (lane == 0) osc[t] = sg16;
    }
  } else {
    // V, one token pair at a time (its rows are interleaved code by code):
    // unit v * (d / 16) + l / 2 holds dims 8l .. 8l + 7 of lanes 2u and 2u + 1
    // for both tokens; the even lane writes words 0 and 1 (its dims 0-3 and
    // 4-7), the odd lane word 2 (its dims 0-3); the odd lane's dims 4-7 fill
    // the bit 3s
    for (int v = warp; v < P / 2; v += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + v * (2 * kHeadDim) + 16 * lane);
      float x0[8], x1[8];
      demote_dequant(__byte_perm(w.x, w.y, 0x6420), __byte_perm(w.z, w.w, 0x6420), __half2float(sc[2 * v]), x0);
      demote_dequant(__byte_perm(w.x, w.y, 0x7531), __byte_perm(w.z, w.w, 0x7531), __half2float(sc[2 * v + 1]), x1);
      __half sg0, sg1;
      const uint32_t n0 = demote_row(x0, sg8, thr, lane, sg0);
      const uint32_t n1 = demote_row(x1, sg8, thr, lane, sg1);
      const uint32_t lo = nibble_zip(n0, n1), hi = nibble_zip(n0 >> 16, n1 >> 16);
      const uint32_t e = __shfl_sync(kFull, hi, lane | 1);
      uint32_t* ud = reinterpret_cast<uint32_t*>(dst + (v * (kHeadDim / 16) + (lane >> 1)) * 12);
      if ((lane & 1) == 0) {
        ud[0] = tq3_word(lo, e, 0);
        ud[1] = tq3_word(hi, e, 1);
      } else {
        ud[2] = tq3_word(lo, e, 2);
      }
      if (lane == 0) {
        osc[2 * v] = sg0;
        osc[2 * v + 1] = sg1;
      }
    }
  }
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

// Code e (0..31) of a 12-byte unit (words w[0..2]).
__device__ __forceinline__ int tq3_unit_code(const uint32_t* w, int e) {
  if (e < 24) return (w[e >> 3] >> (4 * (e & 7))) & 7;
  const int i = e - 24;
  return ((w[0] >> (4 * i + 3)) & 1) | (((w[1] >> (4 * i + 3)) & 1) << 1) | (((w[2] >> (4 * i + 3)) & 1) << 2);
}

// ============================================================== page relevance
// One CTA (4 warps) per (request, page): the page's attention mass, i.e. the
// softmax weight its valid tokens receive averaged over the query heads,
// with each head's weights normalised by the lse of the decode call that
// used the same query: mass = (1/Hq) sum_h sum_t exp(q_h . k_t / sqrt(d) -
// lse_h).  q (or q' = R q for a TQ3 page, whose keys are scored in the
// rotated domain) sits in shared memory; lane l of warp w scores tokens l,
// l + 32, ... of kv head w (and w + 4, ...) against that head's G query
// rows, dequantising each K row as it goes.  Sums reduce in a fixed order.
__global__ void __launch_bounds__(128) mkv_relevance_kernel(RelevanceParams p) {
  extern __shared__ float qs[];                       // [Hq][kHeadDim]
  __shared__ float part[4];
  const int4 pe = p.pages[blockIdx.x];
  const int b = pe.x, page = pe.y, slot = pe.z, tier = pe.w >> 16, nvalid = pe.w & 0xffff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.P;
  // q rows of request b (rotated for a TQ3 page): warp w takes rows w, w + 4, ...
  for (int h = warp; h < p.Hq; h += 4) {
    float x[8];
    const size_t off = (static_cast<size_t>(b) * p.Hq + h) * kHeadDim + 8 * lane;
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
    if (tier == 3) {
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
      for (int i = 0; i < 8; ++i) x[i] *= (1.0f / 16.0f);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) qs[h * kHeadDim + 8 * lane + i] = x[i];
  }
  __syncthreads();
  constexpr float inv_sqrt_d = 1.0f / 16.0f;          // 1 / sqrt(256), exact
  float acc = 0.f;
  for (int kvh = warp; kvh < p.Hkv; kvh += 4) {
    const int rowb = tier == 3 ? 3 * kHeadDim / 8 : kHeadDim;
    const int plane = P * (rowb + 2);
    const uint8_t* kp = (tier == 3 ? p.tq3_layer + static_cast<int64_t>(slot) * p.tq3_page_bytes
                                   : p.fp8_layer + static_cast<int64_t>(slot) * p.fp8_page_bytes) +
                        static_cast<int64_t>(kvh) * 2 * plane;
    const __half* ksc = reinterpret_cast<const __half*>(kp + P * rowb);
    for (int t = lane; t < nvalid; t += 32) {
      const float sc = __half2float(ksc[t]);
      float dot[kMaxGroup];
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) dot[g] = 0.f;
      for (int u = 0; u < kHeadDim / 32; ++u) {        // 32 dims at a time
        float kv[32];
        if (tier == 3) {
          const uint32_t* w = reinterpret_cast<const uint32_t*>(kp + t * rowb + 12 * u);
          const uint32_t wv[3] = {w[0], w[1], w[2]};
#pragma unroll
          for (int e = 0; e < 32; ++e) kv[e] = p.level[tq3_unit_code(wv, e)] * sc;
        } else {
          const uint4* r4 = reinterpret_cast<const uint4*>(kp + t * rowb + 32 * u);
          const uint4 a = r4[0], c = r4[1];
          const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t lo = e4m3x2_to_f16x2(wv[i]), hi = e4m3x2_to_f16x2(wv[i] >> 16);
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            kv[4 * i] = f0.x * sc;
            kv[4 * i + 1] = f0.y * sc;
            kv[4 * i + 2] = f1.x * sc;
            kv[4 * i + 3] = f1.y * sc;
          }
        }
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) {
          if (g < p.G) {
            const float* qr = qs + (kvh * p.G + g) * kHeadDim + 32 * u;
#pragma unroll
            for (int e = 0; e < 32; ++e) dot[g] = fmaf(qr[e], kv[e], dot[g]);
          }
        }
      }
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g)
        if (g < p.G)
          acc += __expf(dot[g] * inv_sqrt_d - p.lse[static_cast<size_t>(b) * p.Hq + kvh * p.G + g]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
  if (lane == 0) part[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0)
    p.mass[static_cast<size_t>(b) * p.mass_stride + page] = ((part[0] + part[1]) + (part[2] + part[3])) / p.Hq;
}

// ============================================================== decode
// Persistent partial-attention kernel; one CTA of 12 warps per SM (8 for
// batch entries of two query tokens).
// The host cut the launch's blocks into one contiguous piece list per CTA,
// minimising the largest CTA's estimated cost (a piece is a run of blocks of
// one (request, kv head, format) group).  Within a piece, warp w takes blocks
// w, w + 12, w + 24, ... and runs the whole of attention on them by itself:
//   S = Q K^T on mma.sync m16n8k16: A = q rows (hi in rows 0-7, lo residual
//     in rows 8-15, fp16), fragments the kernel builds in shared memory for
//     each piece (signs and Walsh-Hadamard rotation for TQ3), B = K dequantised in
//     registers (TQ3: PRMT byte-table lookups; FP8: cvt e4m3x2);
//   online softmax in log2 units with a lazy rescale (per warp);
//   O^T += V^T P^T: A = V dequantised in registers (token pairs), B = P
//     scaled by the V row scales (fp16), the S accumulator layout itself.
// Each warp owns a ring of kSlots shared-memory slots; its lane 0 moves a
// block in with four cp.async.bulk copies (K codes, K scales, V codes, V
// scales) counted by the slot's mbarrier, and refills the slot with the
// warp's block kSlots further on as soon as the warp is done with it.  No
// warp waits for another except at the end of a piece, where the warps'
// states merge, in a fixed order, into one partial state (m, l, o) per q head.
constexpr int kSlotBytes = 2 * (kFp8Blk * kHeadDim + 2 * kFp8Blk);   // an FP8 block; a TQ3 block fits

template <int FMT>
struct Blk {                              // a block of format FMT in a slot
  static constexpr int kTokens = FMT == 0 ? kFp8Blk : kTq3Blk;
  static constexpr int kTiles = kTokens / kTileTokens;
  static constexpr int kRow = FMT == 0 ? kHeadDim : 3 * kHeadDim / 8;      // K row bytes
  static constexpr int kPairRow = 2 * kRow;                                 // V pair-row bytes
  static constexpr int kCode = kTokens * kRow;
  static constexpr int kK = 0, kKs = kCode, kV = kCode + 2 * kTokens, kVs = 2 * kCode + 2 * kTokens;
  static constexpr int kBytes = 2 * (kCode + 2 * kTokens);
};
static_assert(Blk<0>::kBytes <= kSlotBytes && Blk<1>::kBytes <= kSlotBytes, "a block must fit a slot");
static_assert(kSlotBytes % 16 == 0 && Blk<0>::kV % 16 == 0 && Blk<1>::kV % 16 == 0 && Blk<0>::kVs % 16 == 0 &&
                  Blk<1>::kVs % 16 == 0 && Blk<1>::kKs % 16 == 0,
              "bulk copies need 16-byte aligned destinations");

constexpr int kRedBufs = 2;                    // O buffers of the piece-end reduction
constexpr int kRedFloats = 16 * 4 * 32;        // one warp's O fragments, lane-major
constexpr int kQBytes = kQfragWords * 4;       // one piece's q fragments

// CTA shape for NQ query tokens per batch entry (1, or 2 for the paired
// multi-query decode: both queries' O in registers take 8 warps' worth of
// the register file where one query's take 12).
template <int NQ>
struct DecCfg {
  static constexpr int kWarps = dec_warps(NQ);
  static constexpr int kThreads = kWarps * 32;
  // staging slots per warp: 12 x 2 or 8 x 3, 24 blocks in flight per SM
  static constexpr int kSlots = NQ == 1 ? 2 : 3;
  static constexpr int kSmemRing = kWarps * kSlots * kSlotBytes;
  static constexpr int kSmemQ = 2 * NQ * kQBytes;             // [piece i, i+1][query][k-step][lane]
  // the piece-end tree's four buffers: two of their own and the two q
  // buffers (one query token), or the four q buffers (two)
  static constexpr int kSmemRed = NQ == 1 ? kRedBufs * kRedFloats * 4 : 0;
  static constexpr int kSmemEpi = 2 * NQ * kWarps * kMaxGroup * 4;
  static constexpr int kSmemBars = kWarps * kSlots * 8 + 16;
  static constexpr int kSmemBytes = kSmemRing + kSmemQ + kSmemRed + kSmemEpi + kSmemBars;
  static_assert(kSmemBytes <= 227 * 1024, "decode shared memory exceeds the per-CTA limit");
  static_assert(kWarps >= kMaxGroup, "warp h builds row h of a piece's q fragments");
};

struct DecSmem {
  uint8_t* ring;                               // [warp][slot] kSlotBytes
  uint4* qbuf;                                 // [2][NQ][k-step 16][lane 32]: q fragments of pieces i, i+1
  float* red;                                  // [kRedBufs][kRedFloats] (one query token only)
  float* epi_m;                                // [query][warp][kMaxGroup]
  float* epi_l;
  uint64_t* full;                              // [warp][slot]
  int* abort_flag;
};
static_assert(kFp8Blk == 16 && kTq3Blk == 32, "block_locate shifts by log2 of the blocks per 64- or 128-token page");
static_assert(kQBytes == kRedFloats * 4, "a q buffer doubles as a reduction buffer");

template <int NQ>
__device__ __forceinline__ DecSmem dec_carve(uint8_t* base) {
  using C = DecCfg<NQ>;
  DecSmem s;
  s.ring = base;
  s.qbuf = reinterpret_cast<uint4*>(base + C::kSmemRing);
  s.red = reinterpret_cast<float*>(base + C::kSmemRing + C::kSmemQ);
  s.epi_m = reinterpret_cast<float*>(base + C::kSmemRing + C::kSmemQ + C::kSmemRed);
  s.epi_l = s.epi_m + NQ * C::kWarps * kMaxGroup;
  s.full = reinterpret_cast<uint64_t*>(s.epi_l + NQ * C::kWarps * kMaxGroup);
  s.abort_flag = reinterpret_cast<int*>(s.full + C::kWarps * C::kSlots);
  return s;
}

__device__ __forceinline__ bool aborted(const DecSmem& sm) {
  return *reinterpret_cast<volatile int*>(sm.abort_flag) != 0;
}
// Bounded wait (kWaitCycles); gives up at once when the CTA has aborted.
__device__ __forceinline__ bool dec_wait(const DecSmem& sm, uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (aborted(sm)) return false;
    if (mbar_try_wait(bar, parity)) return true;
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

struct Piece {                                 // one CTA piece (its Segment)
  int fmt, b, kvh, entry0, blk0, nblk, part;
};
__device__ __forceinline__ Piece piece_of(const Segment& s) {
  return Piece{s.fmt, s.b, s.kvh, s.entry0, s.blk, s.nblk, s.part};
}
// Piece si of this CTA: the first one travels in the kernel parameters.
__device__ __forceinline__ Piece load_piece(const DecodeParams& p, int si) {
  if (p.heads) return piece_of(p.segs[si]);
  return si == p.cta_seg[blockIdx.x] ? piece_of(p.first[blockIdx.x]) : piece_of(p.segs[si]);
}

// Block k of a piece: page entry, first token within the page, valid tokens
// (<= 0: the block is empty).
__device__ __forceinline__ int block_locate(const DecodeParams& p, const Piece& pc, int k, int& e, int& tok0) {
  const int bt = pc.fmt ? kTq3Blk : kFp8Blk;
  // blocks per page P / bt is a power of two (P is 64 or 128, bt 16 or 32):
  // shift and mask instead of a division by a run-time value
  const int lg = (p.P == 128 ? 3 : 2) - (pc.fmt ? 1 : 0);
  const int bb = pc.blk0 + k;
  e = pc.entry0 + (bb >> lg);
  tok0 = (bb & ((1 << lg) - 1)) * bt;
  return min(bt, static_cast<int>(p.entries[e].nvalid) - tok0);
}

// The warp's sequence of blocks over the CTA's pieces (block k of piece si,
// k = warp, warp + W, ... for W warps).  Every lane keeps the same cursor.
template <int W>
struct BlockCursor {
  int si, s1, k;
  int issued;              // lane 0: blocks copied in so far
  Piece pc;
  __device__ void start(const DecodeParams& p, int s0, int s1_, int warp) {
    issued = 0;
    si = s0;
    s1 = s1_;
    k = warp;
    if (si < s1) pc = load_piece(p, si);
    settle(p, warp);
  }
  __device__ void settle(const DecodeParams& p, int warp) {
    while (si < s1 && k >= pc.nblk) {
      if (++si < s1) pc = load_piece(p, si);
      k = warp;
    }
  }
  __device__ bool valid() const { return si < s1; }
  __device__ void advance(const DecodeParams& p, int warp) {
    k += W;
    settle(p, warp);
  }
};

// Lane 0: copy a block (page entry pe, first token tok0, nv valid tokens) of
// piece pc into slot st (mbarrier bar), or complete the slot's phase without
// bytes for an empty block or a bad plan entry.  Inlined, per format: as an
// out-of-line call it cost 5 % of the kernel (the call once per block).
template <int FMT>
__device__ __forceinline__ void dec_issue_fmt(const DecodeParams& p, const Piece& pc, PageEntry pe, int tok0, int nv,
                                              uint8_t* st, uint64_t* bar, int* abort_flag) {
  const int nslots = FMT ? p.tq3_slots : p.fp8_slots;
  if (nv <= 0) {
    mbar_arrive(bar);
    return;
  }
  if (pe.slot < 0 || pe.slot >= nslots) {
    atomicOr(p.err, kErrBadPlan);
    *reinterpret_cast<volatile int*>(abort_flag) = 1;
    mbar_arrive(bar);
    return;
  }
  constexpr int row = FMT ? 3 * kHeadDim / 8 : kHeadDim;
  constexpr int bt = FMT ? kTq3Blk : kFp8Blk;
  const int plane = p.P * (row + 2);
  const uint8_t* hp = (FMT ? p.tq3_layer : p.fp8_layer) +
                      static_cast<int64_t>(pe.slot) * (FMT ? p.tq3_page_bytes : p.fp8_page_bytes) +
                      static_cast<int64_t>(pc.kvh) * 2 * plane;
  constexpr uint32_t code = bt * row;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, 2 * (code + 2 * bt));
  const uint64_t pol = l2_evict_first_policy();
  bulk_g2s_hint(st, hp + tok0 * row, code, bar, pol);
  bulk_g2s_hint(st + code, hp + p.P * row + 2 * tok0, 2 * bt, bar, pol);
  bulk_g2s_hint(st + code + 2 * bt, hp + plane + tok0 * row, code, bar, pol);
  bulk_g2s_hint(st + 2 * code + 2 * bt, hp + plane + p.P * row + 2 * tok0, 2 * bt, bar, pol);
}
__device__ __forceinline__ void dec_issue_entry(const DecodeParams& p, const Piece& pc, PageEntry pe, int tok0, int nv,
                                                uint8_t* st, uint64_t* bar, int* abort_flag) {
  if (pc.fmt)
    dec_issue_fmt<1>(p, pc, pe, tok0, nv, st, bar, abort_flag);
  else
    dec_issue_fmt<0>(p, pc, pe, tok0, nv, st, bar, abort_flag);
}

// Lane 0: locate block k of piece pc and copy it into slot st.
__device__ __forceinline__ void dec_issue(const DecodeParams& p, const Piece& pc, int k, uint8_t* st, uint64_t* bar,
                                          int* abort_flag) {
  int e = 0, tok0 = 0;
  const int nv = block_locate(p, pc, k, e, tok0);
  dec_issue_entry(p, pc, p.entries[e], tok0, nv, st, bar, abort_flag);
}

// Raw q row h of query token s of piece pc (8 dims per lane, bf16 in r[0]
// or fp32 in r[0..1]); zeros for h >= G.  Split from dec_build_q_row so the
// load can be issued a piece ahead.
struct QRow {
  uint4 r[2];
};
__device__ __forceinline__ QRow dec_load_q_row(const DecodeParams& p, const Piece& pc, int s, int h, int lane) {
  QRow q{};
  if (h < p.G) {
    const int row = q_row(pc.b, s, p.qpe, p.nq, p.npair);
    const size_t off = (static_cast<size_t>(row) * p.Hq + pc.kvh * p.G + h) * kHeadDim + 8 * lane;
    if (p.q_bf16) {
      q.r[0] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + off);
    } else {
      const uint4* f4 = reinterpret_cast<const uint4*>(static_cast<const float*>(p.q) + off);
      q.r[0] = f4[0];
      q.r[1] = f4[1];
    }
  } else {
    q.r[0] = q.r[1] = make_uint4(0u, 0u, 0u, 0u);
  }
  return q;
}

// Row h of piece pc's A fragments from its raw q row, written by one warp
// into q buffer qb: rows 0-7 hold fp16(x), rows 8-15 the fp16 residual
// x - fp16(x), where x is q (FP8 pieces) or q' = R q = (H D q)/16 (TQ3
// pieces; signs, then the Walsh-Hadamard butterflies, 8 dims per lane in
// registers and across lanes by shuffles).  Fragment layout [k-step 16]
// [lane 32][4 regs]: lane (g, c) at k-step j covers dims 64c + 4j .. +3 of
// row g, so lane l of this warp (dims 8l .. 8l+7) fills fragment lane
// 4h + l/8 at k-steps 2(l%8) and 2(l%8) + 1.
__device__ __forceinline__ void dec_build_q_row(const DecodeParams& p, uint4* qb, const Piece& pc, int h, int lane,
                                                const QRow& q, uint32_t qsign) {
  float x[8];
  if (p.q_bf16) {
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&q.r[0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(b2[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else {
    const float* f = reinterpret_cast<const float*>(&q.r[0]);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = f[i];
  }
  if (pc.fmt) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((qsign >> i) & 1u) x[i] = -x[i];
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
    for (int i = 0; i < 8; ++i) x[i] *= (1.0f / 16.0f);
  }
  // the score scale log2(e)/sqrt(d) goes into q here, once per piece, so the
  // scores come out of the MMAs already in log2 units
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] *= p.score_scale;
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    float hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      hi[i] = __half2float(__float2half_rn(x[4 * jj + i]));
      lo[i] = x[4 * jj + i] - hi[i];
    }
    qb[(2 * (lane & 7) + jj) * 32 + 4 * h + (lane >> 3)] =
        make_uint4(pack_half2(hi[0], hi[1]), pack_half2(lo[0], lo[1]), pack_half2(hi[2], hi[3]),
                   pack_half2(lo[2], lo[3]));
  }
}

// The two 12-byte units at p (8-byte aligned): words of unit 0 in u[0..2],
// unit 1 in u[3..5], read as three aligned 8-byte loads.
__device__ __forceinline__ void load_unit_pair(const uint8_t* p, uint32_t (&u)[6]) {
  const uint2 a = *reinterpret_cast<const uint2*>(p);
  const uint2 b = *reinterpret_cast<const uint2*>(p + 8);
  const uint2 c = *reinterpret_cast<const uint2*>(p + 16);
  u[0] = a.x; u[1] = a.y; u[2] = b.x; u[3] = b.y; u[4] = c.x; u[5] = c.y;
}

// S for the one 16-token tile of an FP8 block (two n8 halves: tokens g and
// 8+g as B columns) and each of the NQ query tokens; K rows are row-major,
// the thread's 64 dims are 64 bytes.  A (q) comes k-step by k-step from
// shared memory; each dequantised K fragment feeds every query's MMAs.
template <int NQ>
__device__ __forceinline__ void dec_qk_fp8(const uint8_t* kt, int g, int c, const uint4* const (&qs)[NQ],
                                           float (&s)[NQ][2][2][4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint4 w0 = *reinterpret_cast<const uint4*>(kt + g * kHeadDim + 64 * c + 16 * q4);
    const uint4 w1 = *reinterpret_cast<const uint4*>(kt + (8 + g) * kHeadDim + 64 * c + 16 * q4);
    const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w};
    const uint32_t x1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t b00 = e4m3x2_to_f16x2(x0[i]), b01 = e4m3x2_to_f16x2(x0[i] >> 16);
      const uint32_t b10 = e4m3x2_to_f16x2(x1[i]), b11 = e4m3x2_to_f16x2(x1[i] >> 16);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const uint4 a = qs[q][(4 * q4 + i) * 32 + lane];
        mma16816(s[q][0][0], a.x, a.y, a.z, a.w, b00, b01);
        mma16816(s[q][0][1], a.x, a.y, a.z, a.w, b10, b11);
      }
    }
  }
}

// S for the two 16-token tiles of a TQ3 block: tile t, row (16t + 8r + g),
// units 2c, 2c+1 (24 bytes at 24c).  Each k-step's A fragment is read once
// per query token and feeds the four MMAs (two tiles x two n8 halves); each
// dequantised K fragment feeds every query's MMAs.
template <int NQ>
__device__ __forceinline__ void dec_qk_tq3(const uint8_t* kb, int g, int c, const uint4* const (&qs)[NQ],
                                           const Lut& lut, float (&s)[NQ][2][2][4]) {
  const int lane = threadIdx.x & 31;
  uint32_t u[2][2][6];
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int r = 0; r < 2; ++r) load_unit_pair(kb + (16 * t + 8 * r + g) * 96 + 24 * c, u[t][r]);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t sel[2][2][8];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r)
        tq3_unit_selectors(u[t][r][3 * half], u[t][r][3 * half + 1], u[t][r][3 * half + 2], sel[t][r]);
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      uint4 a[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) a[q] = qs[q][(8 * half + st) * 32 + lane];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint32_t x0, x1;
          tq3_lookup4(sel[t][r][st], lut, x0, x1);
#pragma unroll
          for (int q = 0; q < NQ; ++q) mma16816(s[q][t][r], a[q].x, a[q].y, a[q].z, a[q].w, x0, x1);
        }
    }
  }
}

// O^T += V^T P^T for FP8 V: pair-rows c and c+4 of the tile, dims [32g, 32g+32);
// each dequantised V fragment feeds every query's MMA.
template <int NQ>
__device__ __forceinline__ void dec_pv_fp8(const uint8_t* vt, int g, int c, const uint2 (&pb)[NQ],
                                           float (&o)[NQ][16][4]) {
  const uint8_t* ra = vt + c * (2 * kHeadDim) + 64 * g;
  const uint8_t* rb = vt + (c + 4) * (2 * kHeadDim) + 64 * g;
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint4 wa = *reinterpret_cast<const uint4*>(ra + 16 * q4);
    const uint4 wb = *reinterpret_cast<const uint4*>(rb + 16 * q4);
    const uint32_t xa[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t xb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a0 = e4m3x2_to_f16x2(xa[i]), a1 = e4m3x2_to_f16x2(xa[i] >> 16);
      const uint32_t a2 = e4m3x2_to_f16x2(xb[i]), a3 = e4m3x2_to_f16x2(xb[i] >> 16);
#pragma unroll
      for (int q = 0; q < NQ; ++q) mma16816(o[q][4 * q4 + i], a0, a1, a2, a3, pb[q].x, pb[q].y);
    }
  }
}

// O^T += V^T P^T for TQ3 V: pair-rows c and c+4, units 2g, 2g+1 (24 bytes at 24g)
template <int NQ>
__device__ __forceinline__ void dec_pv_tq3(const uint8_t* vt, int g, int c, const uint2 (&pb)[NQ], const Lut& lut,
                                           float (&o)[NQ][16][4]) {
  uint32_t ua[6], ub[6];
  load_unit_pair(vt + c * 192 + 24 * g, ua);
  load_unit_pair(vt + (c + 4) * 192 + 24 * g, ub);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t sa[8], sb[8];
    tq3_unit_selectors(ua[3 * half], ua[3 * half + 1], ua[3 * half + 2], sa);
    tq3_unit_selectors(ub[3 * half], ub[3 * half + 1], ub[3 * half + 2], sb);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t x0, x1, y0, y1;
      tq3_lookup4(sa[s], lut, x0, x1);
      tq3_lookup4(sb[s], lut, y0, y1);
#pragma unroll
      for (int q = 0; q < NQ; ++q) mma16816(o[q][8 * half + s], x0, x1, y0, y1, pb[q].x, pb[q].y);
    }
  }
}

// Per-warp running state of a piece, per query token.
template <int NQ>
struct WarpState {
  float o[NQ][16][4];      // O^T fragments: m-tile i rows (dims) 32g+2i, 32g+2i+1; columns heads 2c, 2c+1
  float m_run[NQ], l_run[NQ];  // head g: running max (log2 units) and this lane's share of the sum
};

// One block of format FMT at st (nv valid tokens; query token 0 of a paired
// entry sees nv0 of them): scores, online softmax, PV, for each query token.
template <int FMT, int NQ>
__device__ __forceinline__ void dec_block(const DecodeParams& p, const uint8_t* st, int nv, int nv0,
                                          const uint4* const (&qs)[NQ], WarpState<NQ>& ws) {
  using B = Blk<FMT>;
  constexpr int NT = B::kTiles;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const Lut& lut = p.lut;
  float sacc[NQ][2][2][4];
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int h = 0; h < 2; ++h) sacc[q][t][h][0] = sacc[q][t][h][1] = sacc[q][t][h][2] = sacc[q][t][h][3] = 0.f;
  if (FMT == 0)
    dec_qk_fp8<NQ>(st + B::kK, g, c, qs, sacc);
  else
    dec_qk_tq3<NQ>(st + B::kK, g, c, qs, lut, sacc);
  const __half2* ks = reinterpret_cast<const __half2*>(st + B::kKs);
  const __half2* vs = reinterpret_cast<const __half2*>(st + B::kVs);
  const float vsc = FMT == 0 ? kFp8PScale : 1.f;
  uint2 pb[NT][NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int nvq = q == 0 ? nv0 : nv;
    // lane's tokens in tile t: 16t + 2c + {0, 1} (half 0) and 16t + 8 + 2c + {0, 1} (half 1)
    float sc[NT][4];
    float mt = -INFINITY;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float2 k0 = __half22float2(ks[8 * t + c]), k1 = __half22float2(ks[8 * t + 4 + c]);
      sc[t][0] = (sacc[q][t][0][0] + sacc[q][t][0][2]) * k0.x;
      sc[t][1] = (sacc[q][t][0][1] + sacc[q][t][0][3]) * k0.y;
      sc[t][2] = (sacc[q][t][1][0] + sacc[q][t][1][2]) * k1.x;
      sc[t][3] = (sacc[q][t][1][1] + sacc[q][t][1][3]) * k1.y;
      // rows g >= G of q are zero, so those heads score 0 on every token: they
      // never trigger a rescale, and the piece end drops them (m = -inf)
      if (nvq < B::kTokens) {
        const int tb = 16 * t + 2 * c;
        if (tb >= nvq) sc[t][0] = -INFINITY;
        if (tb + 1 >= nvq) sc[t][1] = -INFINITY;
        if (tb + 8 >= nvq) sc[t][2] = -INFINITY;
        if (tb + 9 >= nvq) sc[t][3] = -INFINITY;
      }
      mt = fmaxf(mt, fmaxf(fmaxf(sc[t][0], sc[t][1]), fmaxf(sc[t][2], sc[t][3])));
    }
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
    if (__any_sync(kFull, mt > ws.m_run[q] + kLazyRescale)) {
      const float m_new = fmaxf(ws.m_run[q], mt);
      const float alpha = (ws.m_run[q] == -INFINITY) ? 0.f : ex2(ws.m_run[q] - m_new);
      ws.m_run[q] = m_new;
      ws.l_run[q] *= alpha;
      // O columns are heads 2c and 2c+1: their factors live in lanes 8c and 8c+4
      const float a0 = __shfl_sync(kFull, alpha, 8 * c), a1 = __shfl_sync(kFull, alpha, 8 * c + 4);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        ws.o[q][i][0] *= a0;
        ws.o[q][i][1] *= a1;
        ws.o[q][i][2] *= a0;
        ws.o[q][i][3] *= a1;
      }
    }
    // m_run stays -inf only for heads g >= G (all their scores -inf); a masked
    // score gives ex2(-inf) = 0, and 0 times a (finite, possibly stale) scale is 0
    const float mref = (ws.m_run[q] == -INFINITY) ? 0.f : ws.m_run[q];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = ex2(sc[t][i] - mref);
      ws.l_run[q] += (pr[0] + pr[1]) + (pr[2] + pr[3]);
      const float2 v0 = __half22float2(vs[8 * t + c]), v1 = __half22float2(vs[8 * t + 4 + c]);
      pb[t][q] = make_uint2(pack_half2(pr[0] * (v0.x * vsc), pr[1] * (v0.y * vsc)),
                            pack_half2(pr[2] * (v1.x * vsc), pr[3] * (v1.y * vsc)));
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    if (FMT == 0)
      dec_pv_fp8<NQ>(st + B::kV + t * (kTileTokens / 2) * B::kPairRow, g, c, pb[t], ws.o);
    else
      dec_pv_tq3<NQ>(st + B::kV + t * (kTileTokens / 2) * B::kPairRow, g, c, pb[t], lut, ws.o);
  }
}

// Store / add one warp's O fragments to / from a reduction buffer: m-tile i
// of lane l as one float4 at [i][l] (conflict-free 16-byte accesses).
__device__ __forceinline__ void red_store(float* buf, const float (&o)[16][4]) {
  const int lane = threadIdx.x & 31;
  float4* b4 = reinterpret_cast<float4*>(buf) + lane;
#pragma unroll
  for (int i = 0; i < 16; ++i) b4[i * 32] = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
}
__device__ __forceinline__ void red_add(const float* buf, float (&o)[16][4]) {
  const int lane = threadIdx.x & 31;
  const float4* b4 = reinterpret_cast<const float4*>(buf) + lane;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 v = b4[i * 32];
    o[i][0] += v.x;
    o[i][1] += v.y;
    o[i][2] += v.z;
    o[i][3] += v.w;
  }
}

// End of a piece: the CTA's warps' states merge into the
// piece's partial state, query token by query token.  Each warp rescales its
// O to the common max of each head; O then sums up a fixed tree (four
// buffers) so the result does not depend on timing; warp 0 writes (m, l, o)
// per q head (heads s G .. s G + G - 1 of the piece's partial state for
// query token s).
template <int NQ>
__device__ __forceinline__ void dec_piece_end(const DecodeParams& p, const DecSmem& sm, const Piece& pc,
                                              WarpState<NQ>& ws, int warp) {
  using C = DecCfg<NQ>;
  constexpr int W = C::kWarps;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int G = p.G;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    float l = ws.l_run[q];
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (c == 0) {
      sm.epi_m[(q * W + warp) * kMaxGroup + g] = (g < G) ? ws.m_run[q] : -INFINITY;
      sm.epi_l[(q * W + warp) * kMaxGroup + g] = (g < G) ? l : 0.f;
    }
  }
  named_bar(1, C::kThreads);
  const float osc = pc.fmt == 0 ? 1.f / kFp8PScale : 1.f;
  // the tree: with n warps holding sums, warps [n - h, n) add into warps
  // [0, h), h = min(4, n / 2): one round per level through four 8 KB buffers
  // (see DecCfg; q buffers are free here: the next piece's q fragments are
  // built only after this merge)
  float* const qf = reinterpret_cast<float*>(sm.qbuf);
  auto buf = [&](int i) {
    if (NQ == 1) return i == 0 ? sm.red : i == 1 ? sm.red + kRedFloats : qf + (i - 2) * kRedFloats;
    return qf + i * kRedFloats;
  };
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const float* em = sm.epi_m + q * W * kMaxGroup;
    const float* el = sm.epi_l + q * W * kMaxGroup;
    float f0, f1, Mg = -INFINITY, Lg = 0.f;
    {
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        M0 = fmaxf(M0, em[w * kMaxGroup + 2 * c]);
        M1 = fmaxf(M1, em[w * kMaxGroup + 2 * c + 1]);
        Mg = fmaxf(Mg, em[w * kMaxGroup + g]);
      }
      const float m0 = em[warp * kMaxGroup + 2 * c], m1 = em[warp * kMaxGroup + 2 * c + 1];
      f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - M0) * osc;
      f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - M1) * osc;
      if (warp == 0 && Mg != -INFINITY) {
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float mw = em[w * kMaxGroup + g];
          if (mw != -INFINITY) Lg += ex2(mw - Mg) * el[w * kMaxGroup + g];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      ws.o[q][i][0] *= f0;
      ws.o[q][i][1] *= f1;
      ws.o[q][i][2] *= f0;
      ws.o[q][i][3] *= f1;
    }
    if (q > 0) named_bar(1, C::kThreads);         // the previous query's tree is done with the buffers
#pragma unroll
    for (int n = W; n > 1;) {
      const int h = min(4, n / 2), lo = n - h;
      const int i = warp - lo;                     // this warp as a source
      if (i >= 0 && i < h) red_store(buf(i), ws.o[q]);
      named_bar(1, C::kThreads);
      if (warp < h) red_add(buf(warp), ws.o[q]);
      n = lo;
      if (n > 1) named_bar(1, C::kThreads);
    }
    if (warp == 0) {
      float* dst = p.part + (static_cast<size_t>(pc.part) * NQ + q) * G * (2 + kHeadDim);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int d = 32 * g + 2 * i;
        if (2 * c < G)
          *reinterpret_cast<float2*>(dst + (2 * c) * (2 + kHeadDim) + 2 + d) = make_float2(ws.o[q][i][0], ws.o[q][i][2]);
        if (2 * c + 1 < G)
          *reinterpret_cast<float2*>(dst + (2 * c + 1) * (2 + kHeadDim) + 2 + d) =
              make_float2(ws.o[q][i][1], ws.o[q][i][3]);
      }
      if (c == 0 && g < G) {
        dst[g * (2 + kHeadDim)] = Mg;
        dst[g * (2 + kHeadDim) + 1] = Lg;
      }
    }
  }
}

// The warp's position in its own ring: slot and phase parity of the next
// block it consumes.
template <int S>
struct RingPos {
  int slot, phase;
  __device__ void step() {
    if (++slot == S) {
      slot = 0;
      phase ^= 1;
    }
  }
};

// Fused append (mkv_append_decode): the warp whose FP8 block holds a
// request's newest token quantises the token's K and V rows, stores them into
// the page (global memory, for later steps) and into the staged block it has
// just received (whose copy predates them).
__device__ __forceinline__ void dec_append_tail(const DecodeParams& p, const Piece& pc, const PageEntry& pe, int tok0,
                                                uint8_t* st, int lane) {
  const int pos = pe.nvalid - 1;
  const size_t row = (static_cast<size_t>(pc.b) * p.Hkv + pc.kvh) * kHeadDim;
  const int plane = p.P * (kHeadDim + 2);
  uint8_t* hp = p.fp8_layer + static_cast<int64_t>(pe.slot) * p.fp8_page_bytes + static_cast<int64_t>(pc.kvh) * 2 * plane;
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    uint32_t c[4];
    __half s16;
    fp8_quantize_row(kv ? p.v : p.k, row, p.kv_bf16, lane, c, s16);
    fp8_store_row(hp + kv * plane, p.P, kv, pos, lane, c, s16);
    fp8_store_row(st + kv * (Blk<0>::kBytes / 2), kFp8Blk, kv, pos - tok0, lane, c, s16);
  }
  __syncwarp();
}

// The warp's blocks of piece number pi (piece pc); `ic` is the cursor of the
// next block to copy in.
template <int FMT, int NQ>
__device__ __forceinline__ void dec_piece(const DecodeParams& p, const DecSmem& sm, const Piece& pc, int pi,
                                          BlockCursor<DecCfg<NQ>::kWarps>& ic, RingPos<DecCfg<NQ>::kSlots>& rp,
                                          int warp, WarpState<NQ>& ws) {
  constexpr int W = DecCfg<NQ>::kWarps, kSlots = DecCfg<NQ>::kSlots;
  const int lane = threadIdx.x & 31;
  const uint4* qs[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) qs[q] = sm.qbuf + ((pi & 1) * NQ + q) * (kQBytes / 16);
  for (int k = warp; k < pc.nblk; k += W) {
    int nv = Blk<FMT>::kTokens, e = 0, tok0 = 0;
    if (FMT == 0) nv = block_locate(p, pc, k, e, tok0);
    const bool ok = dec_wait(sm, sm.full + warp * kSlots + rp.slot, rp.phase, p.err);
    uint8_t* st = sm.ring + (warp * kSlots + rp.slot) * kSlotBytes;
    if (ok && nv > 0) {
      int nv0 = nv;
      if (FMT == 0 && NQ == 1 && p.append) {
        const PageEntry pe = p.entries[e];
        if (pe.tail && pe.nvalid - 1 >= tok0 && pe.nvalid - 1 < tok0 + kFp8Blk) dec_append_tail(p, pc, pe, tok0, st, lane);
      }
      if (FMT == 0 && NQ == 2) {
        // a paired entry's prefix ends at its second query token, which its
        // first query token does not see (the causal mask)
        const PageEntry pe = p.entries[e];
        if (pe.tail == kTailPairLast && tok0 + nv == pe.nvalid) nv0 = nv - 1;
      }
      dec_block<FMT, NQ>(p, st, nv, nv0, qs, ws);
    }
    __syncwarp();
    // the slot is free again: copy in the warp's block kSlots further on
    if (ic.valid()) {
      if (lane == 0 && !aborted(sm)) {
        dec_issue(p, ic.pc, ic.k, sm.ring + (warp * kSlots + rp.slot) * kSlotBytes, sm.full + warp * kSlots + rp.slot,
                  sm.abort_flag);
        ++ic.issued;
      }
      ic.advance(p, warp);
    }
    rp.step();
  }
}

template <int NQ>
__global__ void __launch_bounds__(DecCfg<NQ>::kThreads, 1) mkv_decode_kernel(DecodeParams p) {
  using C = DecCfg<NQ>;
  constexpr int W = C::kWarps, kSlots = C::kSlots;
  extern __shared__ __align__(128) uint8_t smem[];
  const DecSmem sm = dec_carve<NQ>(smem);
  // the CTA's pieces: from the kernel parameters, or (a launch whose
  // parameters must not change between steps, e.g. in a CUDA graph) from the
  // plan region in device memory, which is stable while the kernel runs
  const int s0 = p.heads ? p.heads[blockIdx.x] : p.cta_seg[blockIdx.x];
  const int s1 = p.heads ? p.heads[blockIdx.x + 1] : p.cta_seg[blockIdx.x + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the merge kernel that follows waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the rotation signs of this lane's q dims 8 lane .. 8 lane + 7, loaded
  // before the barrier so that the q build does not wait for them
  const uint32_t qsign = static_cast<uint32_t>(
      (lane < 8 ? p.signs[0] : lane < 16 ? p.signs[1] : lane < 24 ? p.signs[2] : p.signs[3]) >> (8 * (lane & 7))) & 0xFFu;
  if (lane == 0) {
    for (int i = 0; i < kSlots; ++i) mbar_init(sm.full + warp * kSlots + i, 1);
    if (warp == 0) *sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // q and the partial-state workspace belong to the preceding kernels (the
  // previous launch's merge reads the workspace): wait for them first
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // warp h < kMaxGroup builds row h of each piece's q fragments (of every
  // query token); piece s0's row loads go out now, the next piece's at the
  // start of each piece
  const bool q_warp = warp < kMaxGroup;
  BlockCursor<W> ic;
  {
    QRow qr[NQ];
    Piece p0{};
    if (q_warp && s0 < s1) {
      p0 = load_piece(p, s0);
#pragma unroll
      for (int q = 0; q < NQ; ++q) qr[q] = dec_load_q_row(p, p0, q, warp, lane);
    }
    // the warp's first kSlots blocks
    ic.start(p, s0, s1, warp);
    Piece fp[kSlots];
    int fk[kSlots];
    int nfirst = 0;
    for (; nfirst < kSlots && ic.valid(); ++nfirst) {
      fp[nfirst] = ic.pc;
      fk[nfirst] = ic.k;
      ic.advance(p, warp);
    }
    // page-entry loads of the first blocks go out together
    PageEntry pe[kSlots];
    int tok0[kSlots], nv[kSlots];
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kSlots; ++i)
        if (i < nfirst) {
          int e = 0;
          nv[i] = block_locate(p, fp[i], fk[i], e, tok0[i]);
          pe[i] = p.entries[e];
        }
      // the first block now; the rest after the q fragments, so that a full
      // copy queue does not hold the warp's q build back
      if (nfirst > 0)
        dec_issue_entry(p, fp[0], pe[0], tok0[0], nv[0], sm.ring + warp * kSlots * kSlotBytes, sm.full + warp * kSlots,
                        sm.abort_flag);
      ic.issued = nfirst;
    }
    if (q_warp && s0 < s1) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) dec_build_q_row(p, sm.qbuf + q * (kQBytes / 16), p0, warp, lane, qr[q], qsign);
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 1; i < kSlots; ++i)
        if (i < nfirst)
          dec_issue_entry(p, fp[i], pe[i], tok0[i], nv[i], sm.ring + (warp * kSlots + i) * kSlotBytes,
                          sm.full + warp * kSlots + i, sm.abort_flag);
    }
    named_bar(1, C::kThreads);
  }
  RingPos<kSlots> rp{0, 0};
  WarpState<NQ> ws;
  for (int si = s0; si < s1; ++si) {
    const int pi = si - s0;
    const Piece pc = load_piece(p, si);
    const bool prep_next = si + 1 < s1 && q_warp;
    Piece pn{};
    QRow qn[NQ];
    if (prep_next) {
      pn = load_piece(p, si + 1);
#pragma unroll
      for (int q = 0; q < NQ; ++q) qn[q] = dec_load_q_row(p, pn, q, warp, lane);
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
#pragma unroll
      for (int i = 0; i < 16; ++i) ws.o[q][i][0] = ws.o[q][i][1] = ws.o[q][i][2] = ws.o[q][i][3] = 0.f;
      ws.m_run[q] = -INFINITY;
      ws.l_run[q] = 0.f;
    }
    if (pc.fmt)
      dec_piece<1, NQ>(p, sm, pc, pi, ic, rp, warp, ws);
    else
      dec_piece<0, NQ>(p, sm, pc, pi, ic, rp, warp, ws);
    dec_piece_end<NQ>(p, sm, pc, ws, warp);
    // every warp is past piece pi; the other q buffers (piece pi - 1's, free
    // since its end) take piece pi + 1
    if (si + 1 < s1) {
      if (prep_next) {
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          dec_build_q_row(p, sm.qbuf + (((pi + 1) & 1) * NQ + q) * (kQBytes / 16), pn, warp, lane, qn[q], qsign);
      }
      named_bar(1, C::kThreads);
    }
  }
  // on the normal path every copy issued was waited for; after an abort, wait
  // (bounded) for copies still in flight before the CTA exits
  __syncthreads();
  if (aborted(sm) && lane == 0) {
    for (int j = ic.issued > kSlots ? ic.issued - kSlots : 0; j < ic.issued; ++j) {
      const long long t0 = clock64();
      while (!mbar_try_wait(sm.full + warp * kSlots + j % kSlots, (j / kSlots) & 1))
        if (clock64() - t0 > kWaitCycles) break;
    }
  }
}

// ============================================================== merge
// One block (256 threads, thread = dim) per (request, kv head, q head).  Each
// format's partial states merge in one pass with a running (M, L, O) -- the
// online-softmax recurrence, in partial-state order, so the result does not
// depend on timing -- loading eight partials at a time.  The TQ3 partials
// merge in the rotated domain, R^T is applied once (FWHT across the block,
// then the signs and 1/16), the FP8 partials join, and out = O / L,
// lse = (M + log2 L) ln 2.
constexpr int kMergeBatch = 8;
constexpr size_t kMergeSmemCap = 200 * 1024;   // dynamic shared memory a merge block may request (unused)

// Loads of partial states [first + base, + kMergeBatch) of head h at dim d.
struct MergeBatch {
  float m[kMergeBatch], l[kMergeBatch], o[kMergeBatch];
};
__device__ __forceinline__ void merge_load(const float* part, int stride, int h, int first, int base, int count,
                                           int d, MergeBatch& mb) {
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u) {
    if (base + u < count) {
      const float* pj = part + static_cast<size_t>(first + base + u) * stride + h * (2 + kHeadDim);
      mb.m[u] = pj[0];
      mb.l[u] = pj[1];
      mb.o[u] = pj[2 + d];
    } else {
      mb.m[u] = -INFINITY;
      mb.l[u] = 0.f;
      mb.o[u] = 0.f;
    }
  }
}
__device__ __forceinline__ void merge_fold(const MergeBatch& mb, float& M, float& L, float& O) {
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u) {
    if (mb.m[u] == -INFINITY) continue;   // an empty head (the same for every thread)
    const float Mn = fmaxf(M, mb.m[u]);
    const float a = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
    const float w = exp2f(mb.m[u] - Mn);
    L = L * a + mb.l[u] * w;
    O = O * a + mb.o[u] * w;
    M = Mn;
  }
}
// Partial states [first, first + count) of head h merged at dim d; the first
// batch is passed in already loaded.  With PREFETCH the next batch's loads go
// out before the current batch is folded (two batches in flight, more
// registers); the fold order, and so the result, is the same either way.
template <bool PREFETCH>
__device__ __forceinline__ void merge_run(const float* part, int stride, int h, int first, int count, int d,
                                          const MergeBatch& first_batch, float& M, float& L, float& O) {
  M = -INFINITY;
  L = 0.f;
  O = 0.f;
  if (PREFETCH) {
    MergeBatch cur = first_batch;
    for (int base = kMergeBatch; base < count; base += kMergeBatch) {
      MergeBatch nxt;
      merge_load(part, stride, h, first, base, count, d, nxt);
      merge_fold(cur, M, L, O);
      cur = nxt;
    }
    merge_fold(cur, M, L, O);
  } else {
    merge_fold(first_batch, M, L, O);
    for (int base = kMergeBatch; base < count; base += kMergeBatch) {
      MergeBatch mb;
      merge_load(part, stride, h, first, base, count, d, mb);
      merge_fold(mb, M, L, O);
    }
  }
}

template <bool PREFETCH>
__global__ void __launch_bounds__(256) mkv_merge_kernel(MergeParams p) {
  __shared__ float xs[kHeadDim];
  // head h of the entry's partial states: query token h / G, q head h % G
  const int Ge = p.qpe * p.G;
  const int h = blockIdx.x % Ge;
  const int bk = blockIdx.x / Ge;
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  // the merge descriptors come with the plan (copied in before the decode
  // kernel started), so they load while the decode kernel still runs
  const MergeDesc md = p.desc[bk];
  const bool neg = sign_neg(p.signs, threadIdx.x);
  // launched as a programmatic dependent of the decode kernel: wait for its
  // partial states before reading them
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int d = threadIdx.x, lane = d & 31;
  const int stride = Ge * (2 + kHeadDim);
  // the first batch of both formats goes out at once
  MergeBatch bs, bf;
  merge_load(p.part, stride, h, md.tq3_first, 0, md.tq3_count, d, bs);
  merge_load(p.part, stride, h, md.fp8_first, 0, md.fp8_count, d, bf);
  float Ms, Ls, os, Mf, Lf, of;
  merge_run<PREFETCH>(p.part, stride, h, md.tq3_first, md.tq3_count, d, bs, Ms, Ls, os);
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
  if (neg) os = -os;
  merge_run<PREFETCH>(p.part, stride, h, md.fp8_first, md.fp8_count, d, bf, Mf, Lf, of);
  const float M = fmaxf(Ms, Mf);
  const float fs = (Ms == -INFINITY) ? 0.f : exp2f(Ms - M);
  const float ff = (Mf == -INFINITY) ? 0.f : exp2f(Mf - M);
  const float L = Ls * fs + Lf * ff;
  const int hq = kvh * p.G + h % p.G;
  const int row = q_row(b, h / p.G, p.qpe, p.nq, p.npair);
  p.out[(static_cast<size_t>(row) * p.Hq + hq) * kHeadDim + d] = (os * fs + of * ff) / L;
  if (d == 0) p.lse[row * p.Hq + hq] = (M + log2f(L)) * 0.69314718055994530942f;
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
  if (blocks > 0) mkv_demote_kernel<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

size_t decode_smem_bytes() { return DecCfg<1>::kSmemBytes; }


// Fixed scratch for the allocation-free decode entry point: 8 MiB of partial
// states, compiled into the library so a call never needs to allocate.
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchBytes / sizeof(float)];

cudaError_t noalloc_scratch(float** ptr, size_t* bytes) {
  // looked up on every call (cheap, and not a stream operation): a cached
  // address would dangle after the device's context is reset and rebuilt.
  // Host code must not use the symbol itself as a device address.
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *ptr = static_cast<float*>(p);
  *bytes = kNoallocScratchBytes;
  return cudaSuccess;
}
int decode_threads() { return DecCfg<1>::kThreads; }

cudaError_t launch_relevance(const RelevanceParams& p, cudaStream_t s) {
  if (p.npages > 0)
    mkv_relevance_kernel<<<p.npages, 128, static_cast<size_t>(p.Hq) * kHeadDim * sizeof(float), s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantParams& p, cudaStream_t s) {
  const int rows = p.npages * p.P * p.Hkv * 2;
  if (rows > 0) mkv_dequant_kernel<<<(rows + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t prepare_decode_launch() {
  // the shared-memory limits (the decode kernel's, and the merge kernel's
  // unused request) are per-device attributes: set them once per device
  // (setting them twice from racing threads is harmless)
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(mkv_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DecCfg<1>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mkv_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DecCfg<2>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mkv_merge_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSmemCap);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_acq_rel);
  }
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
  cudaError_t e = prepare_decode_launch();
  if (e != cudaSuccess) return e;
  if (p.n_ctas <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_ctas);
  const bool pair = p.qpe == 2;
  cfg.blockDim = dim3(pair ? DecCfg<2>::kThreads : DecCfg<1>::kThreads);
  cfg.dynamicSmemBytes = pair ? DecCfg<2>::kSmemBytes : DecCfg<1>::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return pair ? cudaLaunchKernelEx(&cfg, mkv_decode_kernel<2>, p) : cudaLaunchKernelEx(&cfg, mkv_decode_kernel<1>, p);
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.n * p.Hkv <= 0) return cudaSuccess;
  // The merge blocks land on SMs as the decode CTAs leave them, so the first
  // SMs to free up would take as many blocks as fit; an unused dynamic
  // shared-memory request caps the blocks per SM at what spreads the grid
  // over all SMs in one wave.  At one or two blocks per SM the registers of
  // the prefetching variant cost no occupancy, so that variant runs.
  // (the kernel's shared-memory limit is raised by prepare_decode_launch,
  // which every decode launch, and a graph capture, runs first)
  int dev = 0, n_sm = 0, smem_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  const int grid = p.n * p.Hkv * p.qpe * p.G;
  const int per_sm = (grid + n_sm - 1) / n_sm;
  size_t dyn = 0;
  if (per_sm <= 2) {
    dyn = static_cast<size_t>(smem_sm / per_sm - 4096);
    if (dyn > kMergeSmemCap) dyn = kMergeSmemCap;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kHeadDim);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return per_sm <= 2 ? cudaLaunchKernelEx(&cfg, mkv_merge_kernel<true>, p)
                     : cudaLaunchKernelEx(&cfg, mkv_merge_kernel<false>, p);
}

}  // namespace mkv
