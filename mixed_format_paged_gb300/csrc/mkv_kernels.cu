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
//   mkv_decode_kernel  -- persistent partial-attention kernel; CTAs below
//                         n_ctas_fp8 run the FP8 body, the rest the TQ3 body
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
// Bounded wait: false when the phase did not complete within kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
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
  return (signs[i >> 6] >> (i & 63)) & 1ull;
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
// One warp per (token, kv head, K|V) row: FP8 scale + codes into the page.
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
  const size_t row = (static_cast<size_t>(tok) * p.Hkv + h) * kHeadDim;
  const void* src = kv ? p.v : p.k;
  float x[8];
  if (p.kv_bf16) {
    const uint4 raw = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + row)[lane];
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(b2[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else {
    const float4* f4 = reinterpret_cast<const float4*>(static_cast<const float*>(src) + row) + 2 * lane;
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
  const int P = p.P;
  uint8_t* plane = p.fp8_layer + static_cast<int64_t>(slot) * p.fp8_page_bytes +
                   static_cast<int64_t>(h) * 2 * (P * (kHeadDim + 2)) + kv * (P * (kHeadDim + 2));
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

// ============================================================== decode
// Persistent partial-attention kernel.  Warps 0..7 consume, warp 8 produces.
//
// Producer: for every 64-token block of every page of the CTA's chunks, one
// mbarrier-tracked cp.async.bulk per plane part (K codes, K scales, V codes,
// V scales) into a ring of kStages(fmt) shared-memory stages.
// Consumers: warps 0-3 take even blocks and warps 4-7 odd ones; warp w owns
// tokens [16 (w%4), +16) of its block.  Per 16-token tile:
//   S^T = Q K^T on mma.sync m16n8k16: A = q rows (hi in rows 0-7, lo
//   residual in rows 8-15, fp16) from registers, B = dequantised K;
//   online softmax in log2 units with a lazy rescale;
//   O^T += V^T P^T: A = dequantised V (token pairs), B = P scaled by the
//   V row scales (fp16).
// Epilogue per chunk: the 8 warps' states merge in shared memory into one
// partial (m, l, o) per q head.
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {  // FP8
  static constexpr int kRowBytes = kHeadDim;            // K row / half V pair-row
  static constexpr int kStages = 4;
};
template <>
struct Fmt<1> {  // TQ3
  static constexpr int kRowBytes = 3 * kHeadDim / 8;
  static constexpr int kStages = 10;
};
template <int FMT>
struct Stage {
  static constexpr int kCode = kStageTokens * Fmt<FMT>::kRowBytes;    // bytes of K (or V) codes
  static constexpr int kScale = kStageTokens * 2;
  static constexpr int kK = 0, kKs = kCode, kV = kCode + kScale, kVs = 2 * kCode + kScale;
  static constexpr int kBytes = 2 * (kCode + kScale);
};

constexpr int kEpiFloats = kConsumerWarps * kMaxGroup * kHeadDim;     // O per warp
constexpr int kSmemRing = 4 * Stage<0>::kBytes > 10 * Stage<1>::kBytes ? 4 * Stage<0>::kBytes
                                                                       : 10 * Stage<1>::kBytes;
constexpr int kSmemBytes = kSmemRing + kEpiFloats * 4 + 2 * kConsumerWarps * kMaxGroup * 4 +
                           kMaxGroup * kHeadDim * 4 + 2 * 16 * 8 + 64;

struct SmemLayout {
  uint8_t* ring;
  float* epi_o;   // [warp][head][D]
  float* epi_m;   // [warp][head]
  float* epi_l;
  float* qs;      // [head][D]
  uint64_t* full;
  uint64_t* empty;
  int* abort_flag;
};
__device__ __forceinline__ SmemLayout carve(uint8_t* base) {
  SmemLayout s;
  s.ring = base;
  s.epi_o = reinterpret_cast<float*>(base + kSmemRing);
  s.epi_m = s.epi_o + kEpiFloats;
  s.epi_l = s.epi_m + kConsumerWarps * kMaxGroup;
  s.qs = s.epi_l + kConsumerWarps * kMaxGroup;
  s.full = reinterpret_cast<uint64_t*>(s.qs + kMaxGroup * kHeadDim);
  s.empty = s.full + 16;
  s.abort_flag = reinterpret_cast<int*>(s.empty + 16);
  return s;
}

// number of 64-token blocks of a page entry that hold valid tokens
__device__ __forceinline__ int entry_blocks(const PageEntry& e) {
  return (e.nvalid + kStageTokens - 1) / kStageTokens;
}

template <int FMT>
__device__ void producer_loop(const DecodeParams& p, const SmemLayout& sm, int first, int last) {
  using St = Stage<FMT>;
  constexpr int NS = Fmt<FMT>::kStages;
  const uint8_t* arena = FMT == 0 ? p.fp8_layer : p.tq3_layer;
  const int64_t page_bytes = FMT == 0 ? p.fp8_page_bytes : p.tq3_page_bytes;
  const int nslots = FMT == 0 ? p.fp8_slots : p.tq3_slots;
  const int P = p.P;
  const int plane = P * (Fmt<FMT>::kRowBytes + 2);
  int gi = 0;   // global block counter
  bool ok = true;
  for (int ci = first; ci < last && ok; ++ci) {
    const Chunk ch = p.chunks[p.cta_chunks[ci]];
    for (int e = 0; e < ch.nentry && ok; ++e) {
      const PageEntry pe = p.entries[ch.entry0 + e];
      if (pe.slot < 0 || pe.slot >= nslots) {
        atomicOr(p.err, kErrBadPlan);
        ok = false;
        break;
      }
      const uint8_t* hp = arena + static_cast<int64_t>(pe.slot) * page_bytes +
                          static_cast<int64_t>(ch.kvh) * 2 * plane;
      const int nb = entry_blocks(pe);
      for (int blk = 0; blk < nb; ++blk, ++gi) {
        const int slot = gi % NS;
        if (gi >= NS) {
          if (!mbar_wait(&sm.empty[slot], ((gi / NS) - 1) & 1)) {
            atomicOr(p.err, kErrWaitTimeout);
            *sm.abort_flag = 1;
            ok = false;
            break;
          }
        }
        if (*reinterpret_cast<volatile int*>(sm.abort_flag)) { ok = false; break; }
        uint8_t* st = sm.ring + slot * St::kBytes;
        const int tok0 = blk * kStageTokens;
        mbar_expect_tx(&sm.full[slot], St::kBytes);
        bulk_g2s(st + St::kK, hp + tok0 * Fmt<FMT>::kRowBytes, St::kCode, &sm.full[slot]);
        bulk_g2s(st + St::kKs, hp + P * Fmt<FMT>::kRowBytes + tok0 * 2, St::kScale, &sm.full[slot]);
        bulk_g2s(st + St::kV, hp + plane + tok0 * Fmt<FMT>::kRowBytes, St::kCode, &sm.full[slot]);
        bulk_g2s(st + St::kVs, hp + plane + P * Fmt<FMT>::kRowBytes + tok0 * 2, St::kScale, &sm.full[slot]);
      }
    }
  }
  // drain: wait (bounded) for every issued copy so none lands after exit
  for (int k = (gi > NS ? gi - NS : 0); k < gi; ++k) {
    const int slot = k % NS;
    if (!mbar_wait(&sm.full[slot], (k / NS) & 1)) {
      atomicOr(p.err, kErrWaitTimeout);
      break;
    }
  }
}

// Q prologue: q rows of this (b, kvh) -> fp32 in smem (rotated for TQ3) ->
// per-warp A fragments (hi / lo fp16).
template <int FMT>
__device__ __forceinline__ void load_q_frags(const DecodeParams& p, const SmemLayout& sm, int b, int kvh,
                                             uint32_t (&qa)[16][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // warp w loads head w (zero when w >= G)
  {
    float x[8];
    const int hq = kvh * p.G + warp;
    if (warp < p.G) {
      const size_t off = (static_cast<size_t>(b) * p.Hq + hq) * kHeadDim + 8 * lane;
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
    if (FMT == 1) {   // q' = R q = H (signs .* q) / 16
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
    float4* dst = reinterpret_cast<float4*>(sm.qs + warp * kHeadDim + 8 * lane);
    dst[0] = make_float4(x[0], x[1], x[2], x[3]);
    dst[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
  named_bar(1, kConsumerWarps * 32);
  const int g = lane >> 2, c = lane & 3;
  const float* qr = sm.qs + g * kHeadDim + 64 * c;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float4 v = *reinterpret_cast<const float4*>(qr + 4 * j);
    const float vv[4] = {v.x, v.y, v.z, v.w};
    float hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      hi[i] = __half2float(__float2half_rn(vv[i]));
      lo[i] = vv[i] - hi[i];
    }
    qa[j][0] = pack_half2(hi[0], hi[1]);
    qa[j][1] = pack_half2(lo[0], lo[1]);
    qa[j][2] = pack_half2(hi[2], hi[3]);
    qa[j][3] = pack_half2(lo[2], lo[3]);
  }
}

// S tile (two n8 halves) for one 16-token tile: FP8 K
__device__ __forceinline__ void qk_fp8(const uint8_t* kbase, int g, int c, const uint32_t (&qa)[16][4],
                                       float (&s0)[4], float (&s1)[4]) {
  float a0[4] = {0, 0, 0, 0}, a1[4] = {0, 0, 0, 0};
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint4 w0 = *reinterpret_cast<const uint4*>(kbase + g * kHeadDim + 64 * c + 16 * q4);
    const uint4 w1 = *reinterpret_cast<const uint4*>(kbase + (8 + g) * kHeadDim + 64 * c + 16 * q4);
    const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w};
    const uint32_t x1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 4 * q4 + i;
      float(&acc0)[4] = (j & 1) ? a0 : s0;
      float(&acc1)[4] = (j & 1) ? a1 : s1;
      mma16816(acc0, qa[j][0], qa[j][1], qa[j][2], qa[j][3], e4m3x2_to_f16x2(x0[i]),
               e4m3x2_to_f16x2(x0[i] >> 16));
      mma16816(acc1, qa[j][0], qa[j][1], qa[j][2], qa[j][3], e4m3x2_to_f16x2(x1[i]),
               e4m3x2_to_f16x2(x1[i] >> 16));
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s0[i] += a0[i];
    s1[i] += a1[i];
  }
}

// S tile for TQ3 K: row (u*8 + g) units 2c, 2c+1 (24 bytes at 24c)
__device__ __forceinline__ void qk_tq3(const uint8_t* kbase, int g, int c, const uint32_t (&qa)[16][4],
                                       const Lut& lut, float (&s0)[4], float (&s1)[4]) {
  float a0[4] = {0, 0, 0, 0}, a1[4] = {0, 0, 0, 0};
  const uint8_t* r0 = kbase + g * 96 + 24 * c;
  const uint8_t* r1 = kbase + (8 + g) * 96 + 24 * c;
  const uint2 p0 = *reinterpret_cast<const uint2*>(r0), p1 = *reinterpret_cast<const uint2*>(r0 + 8),
              p2 = *reinterpret_cast<const uint2*>(r0 + 16);
  const uint2 q0 = *reinterpret_cast<const uint2*>(r1), q1 = *reinterpret_cast<const uint2*>(r1 + 8),
              q2 = *reinterpret_cast<const uint2*>(r1 + 16);
  const uint32_t wa[6] = {p0.x, p0.y, p1.x, p1.y, p2.x, p2.y};
  const uint32_t wb[6] = {q0.x, q0.y, q1.x, q1.y, q2.x, q2.y};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t sa[8], sb[8];
    tq3_unit_selectors(wa[3 * half], wa[3 * half + 1], wa[3 * half + 2], sa);
    tq3_unit_selectors(wb[3 * half], wb[3 * half + 1], wb[3 * half + 2], sb);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int j = 8 * half + s;
      uint32_t b0, b1, d0, d1;
      tq3_lookup4(sa[s], lut, b0, b1);
      tq3_lookup4(sb[s], lut, d0, d1);
      float(&acc0)[4] = (j & 1) ? a0 : s0;
      float(&acc1)[4] = (j & 1) ? a1 : s1;
      mma16816(acc0, qa[j][0], qa[j][1], qa[j][2], qa[j][3], b0, b1);
      mma16816(acc1, qa[j][0], qa[j][1], qa[j][2], qa[j][3], d0, d1);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s0[i] += a0[i];
    s1[i] += a1[i];
  }
}

// O^T += V^T P^T for FP8 V: pair-rows c and c+4 of the tile, dims [32g, 32g+32)
__device__ __forceinline__ void pv_fp8(const uint8_t* vbase, int g, int c, uint32_t pb0, uint32_t pb1,
                                       float (&o)[16][4]) {
  const uint8_t* ra = vbase + c * (2 * kHeadDim) + 64 * g;
  const uint8_t* rb = vbase + (c + 4) * (2 * kHeadDim) + 64 * g;
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint4 wa = *reinterpret_cast<const uint4*>(ra + 16 * q4);
    const uint4 wb = *reinterpret_cast<const uint4*>(rb + 16 * q4);
    const uint32_t xa[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t xb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int mt = 4 * q4 + i;
      mma16816(o[mt], e4m3x2_to_f16x2(xa[i]), e4m3x2_to_f16x2(xa[i] >> 16), e4m3x2_to_f16x2(xb[i]),
               e4m3x2_to_f16x2(xb[i] >> 16), pb0, pb1);
    }
  }
}

// O^T += V^T P^T for TQ3 V: pair-rows c and c+4, units 2g, 2g+1 (24 bytes at 24g)
__device__ __forceinline__ void pv_tq3(const uint8_t* vbase, int g, int c, uint32_t pb0, uint32_t pb1,
                                       const Lut& lut, float (&o)[16][4]) {
  const uint8_t* ra = vbase + c * 192 + 24 * g;
  const uint8_t* rb = vbase + (c + 4) * 192 + 24 * g;
  const uint2 p0 = *reinterpret_cast<const uint2*>(ra), p1 = *reinterpret_cast<const uint2*>(ra + 8),
              p2 = *reinterpret_cast<const uint2*>(ra + 16);
  const uint2 q0 = *reinterpret_cast<const uint2*>(rb), q1 = *reinterpret_cast<const uint2*>(rb + 8),
              q2 = *reinterpret_cast<const uint2*>(rb + 16);
  const uint32_t wa[6] = {p0.x, p0.y, p1.x, p1.y, p2.x, p2.y};
  const uint32_t wb[6] = {q0.x, q0.y, q1.x, q1.y, q2.x, q2.y};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t sa[8], sb[8];
    tq3_unit_selectors(wa[3 * half], wa[3 * half + 1], wa[3 * half + 2], sa);
    tq3_unit_selectors(wb[3 * half], wb[3 * half + 1], wb[3 * half + 2], sb);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t a0, a1, a2, a3;
      tq3_lookup4(sa[s], lut, a0, a1);
      tq3_lookup4(sb[s], lut, a2, a3);
      mma16816(o[8 * half + s], a0, a1, a2, a3, pb0, pb1);
    }
  }
}

template <int FMT>
__device__ void consumer_loop(const DecodeParams& p, const SmemLayout& sm, int first, int last) {
  using St = Stage<FMT>;
  constexpr int NS = Fmt<FMT>::kStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int grp = warp >> 2, tile = warp & 3;
  const Lut lut = p.lut;
  const int G = p.G;
  uint32_t qa[16][4];
  float o[16][4];
  int gi = 0;
  for (int ci = first; ci < last; ++ci) {
    const int cid = p.cta_chunks[ci];
    const Chunk ch = p.chunks[cid];
    load_q_frags<FMT>(p, sm, ch.b, ch.kvh, qa);
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;   // head g, per-thread partial l
    bool aborted = false;
    for (int e = 0; e < ch.nentry && !aborted; ++e) {
      const PageEntry pe = p.entries[ch.entry0 + e];
      const int nb = entry_blocks(pe);
      for (int blk = 0; blk < nb; ++blk, ++gi) {
        if ((gi & 1) != grp) continue;
        const int slot = gi % NS;
        if (!mbar_wait(&sm.full[slot], (gi / NS) & 1)) {
          atomicOr(p.err, kErrWaitTimeout);
          *sm.abort_flag = 1;
          aborted = true;
          break;
        }
        const int base = blk * kStageTokens + tile * kTileTokens;   // first token of this tile in the page
        const int nv = pe.nvalid - base;
        if (nv > 0) {
          const uint8_t* st = sm.ring + slot * St::kBytes;
          float s0[4] = {0, 0, 0, 0}, s1[4] = {0, 0, 0, 0};
          if (FMT == 0)
            qk_fp8(st + St::kK + tile * kTileTokens * kHeadDim, g, c, qa, s0, s1);
          else
            qk_tq3(st + St::kK + tile * kTileTokens * 96, g, c, qa, lut, s0, s1);
          // scores of head g at tokens 2c, 2c+1, 8+2c, 9+2c (log2 units)
          const __half2* ks = reinterpret_cast<const __half2*>(st + St::kKs + tile * kTileTokens * 2);
          const __half2* vs = reinterpret_cast<const __half2*>(st + St::kVs + tile * kTileTokens * 2);
          const float2 k01 = __half22float2(ks[c]), k89 = __half22float2(ks[4 + c]);
          const float2 v01 = __half22float2(vs[c]), v89 = __half22float2(vs[4 + c]);
          float sc[4];
          sc[0] = (s0[0] + s0[2]) * k01.x * p.score_scale;
          sc[1] = (s0[1] + s0[3]) * k01.y * p.score_scale;
          sc[2] = (s1[0] + s1[2]) * k89.x * p.score_scale;
          sc[3] = (s1[1] + s1[3]) * k89.y * p.score_scale;
          const int tk[4] = {2 * c, 2 * c + 1, 8 + 2 * c, 9 + 2 * c};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (tk[i] >= nv || g >= G) sc[i] = -INFINITY;
          float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
          mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
          mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
          const bool need = mt > m_run + kLazyRescale;
          if (__any_sync(kFull, need)) {
            const float m_new = fmaxf(m_run, mt);
            const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
            m_run = m_new;
            l_run *= alpha;
            const float a0 = __shfl_sync(kFull, alpha, (2 * c) * 4);
            const float a1 = __shfl_sync(kFull, alpha, (2 * c + 1) * 4);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              o[i][0] *= a0;
              o[i][1] *= a1;
              o[i][2] *= a0;
              o[i][3] *= a1;
            }
          }
          float pr[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) pr[i] = (sc[i] == -INFINITY) ? 0.f : exp2f(sc[i] - m_run);
          l_run += (pr[0] + pr[1]) + (pr[2] + pr[3]);
          const float vsc = FMT == 0 ? kFp8PScale : 1.0f;
          const uint32_t pb0 = pack_half2(pr[0] * v01.x * vsc, pr[1] * v01.y * vsc);
          const uint32_t pb1 = pack_half2(pr[2] * v89.x * vsc, pr[3] * v89.y * vsc);
          if (FMT == 0)
            pv_fp8(st + St::kV + tile * (kTileTokens / 2) * (2 * kHeadDim), g, c, pb0, pb1, o);
          else
            pv_tq3(st + St::kV + tile * (kTileTokens / 2) * 192, g, c, pb0, pb1, lut, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }
    }
    // ---- epilogue: merge the 8 warps' states into one partial
    l_run += __shfl_xor_sync(kFull, l_run, 1);
    l_run += __shfl_xor_sync(kFull, l_run, 2);
    if (c == 0) {
      sm.epi_m[warp * kMaxGroup + g] = m_run;
      sm.epi_l[warp * kMaxGroup + g] = l_run;
    }
    const float osc = FMT == 0 ? 1.0f / kFp8PScale : 1.0f;
    float* ow = sm.epi_o + warp * kMaxGroup * kHeadDim;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int d = 32 * g + 2 * i;
      *reinterpret_cast<float2*>(ow + (2 * c) * kHeadDim + d) = make_float2(o[i][0] * osc, o[i][2] * osc);
      *reinterpret_cast<float2*>(ow + (2 * c + 1) * kHeadDim + d) = make_float2(o[i][1] * osc, o[i][3] * osc);
    }
    named_bar(1, kConsumerWarps * 32);
    {
      const int d = threadIdx.x;   // 0..255
      float* dst = p.part + static_cast<size_t>(cid) * G * (2 + kHeadDim);
      for (int h = 0; h < G; ++h) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.epi_m[w * kMaxGroup + h]);
        float L = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = sm.epi_m[w * kMaxGroup + h];
            const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            L += f * sm.epi_l[w * kMaxGroup + h];
            acc += f * sm.epi_o[(w * kMaxGroup + h) * kHeadDim + d];
          }
        }
        dst[h * (2 + kHeadDim) + 2 + d] = acc;
        if (d == 0) {
          dst[h * (2 + kHeadDim)] = M;
          dst[h * (2 + kHeadDim) + 1] = L;
        }
      }
    }
    named_bar(1, kConsumerWarps * 32);
    if (aborted || *reinterpret_cast<volatile int*>(sm.abort_flag)) return;
  }
}

template <int FMT>
__device__ void decode_body(const DecodeParams& p, const SmemLayout& sm, int first, int last) {
  const int warp = threadIdx.x >> 5;
  if (warp == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) producer_loop<FMT>(p, sm, first, last);
  } else {
    consumer_loop<FMT>(p, sm, first, last);
  }
}

__global__ void __launch_bounds__(kThreads, 1) mkv_decode_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout sm = carve(smem);
  const int cta = blockIdx.x;
  const int first = p.cta_start[cta], last = p.cta_start[cta + 1];
  const bool fp8 = cta < p.n_ctas_fp8;
  if (threadIdx.x == 0) {
    const int ns = fp8 ? Fmt<0>::kStages : Fmt<1>::kStages;
    for (int i = 0; i < ns; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 4);
    }
    *sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (first >= last) return;
  if (fp8)
    decode_body<0>(p, sm, first, last);
  else
    decode_body<1>(p, sm, first, last);
}

// ============================================================== merge
// One block (256 threads, thread = dim) per (b, kvh).  TQ3 partials merge in
// the rotated domain, R^T is applied once (FWHT across the block), then the
// FP8 partials join; out = O / L, lse = (M + log2 L) ln 2.
__global__ void __launch_bounds__(256) mkv_merge_kernel(MergeParams p) {
  __shared__ float xs[kHeadDim];
  const int b = blockIdx.x / p.Hkv, kvh = blockIdx.x % p.Hkv;
  const MergeDesc md = p.desc[blockIdx.x];
  const int d = threadIdx.x, lane = d & 31;
  const int stride = p.G * (2 + kHeadDim);
  for (int h = 0; h < p.G; ++h) {
    // TQ3 partials
    float Ms = -INFINITY, Ls = 0.f, os = 0.f;
    for (int j = 0; j < md.tq3_count; ++j) Ms = fmaxf(Ms, p.part[(md.tq3_first + j) * stride + h * (2 + kHeadDim)]);
    if (Ms != -INFINITY) {
      for (int j = 0; j < md.tq3_count; ++j) {
        const float* pj = p.part + (md.tq3_first + j) * stride + h * (2 + kHeadDim);
        const float f = (pj[0] == -INFINITY) ? 0.f : exp2f(pj[0] - Ms);
        Ls += f * pj[1];
        os += f * pj[2 + d];
      }
    }
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
    // FP8 partials
    float Mf = -INFINITY, Lf = 0.f, of = 0.f;
    for (int j = 0; j < md.fp8_count; ++j) Mf = fmaxf(Mf, p.part[(md.fp8_first + j) * stride + h * (2 + kHeadDim)]);
    if (Mf != -INFINITY) {
      for (int j = 0; j < md.fp8_count; ++j) {
        const float* pj = p.part + (md.fp8_first + j) * stride + h * (2 + kHeadDim);
        const float f = (pj[0] == -INFINITY) ? 0.f : exp2f(pj[0] - Mf);
        Lf += f * pj[1];
        of += f * pj[2 + d];
      }
    }
    const float M = fmaxf(Ms, Mf);
    const float fs = (Ms == -INFINITY) ? 0.f : exp2f(Ms - M);
    const float ff = (Mf == -INFINITY) ? 0.f : exp2f(Mf - M);
    const float L = Ls * fs + Lf * ff;
    const int hq = kvh * p.G + h;
    p.out[(static_cast<size_t>(b) * p.Hq + hq) * kHeadDim + d] = (os * fs + of * ff) / L;
    if (d == 0) p.lse[b * p.Hq + hq] = (M + log2f(L)) * 0.69314718055994530942f;
    __syncthreads();
  }
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

size_t decode_smem_bytes() { return kSmemBytes; }

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
int decode_threads() { return kThreads; }

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(mkv_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (p.n_ctas > 0) mkv_decode_kernel<<<p.n_ctas, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.n * p.Hkv > 0) mkv_merge_kernel<<<p.n * p.Hkv, kHeadDim, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mkv
