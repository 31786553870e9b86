// Device helpers shared by the kernels of mkv_kernels.cu and mkv_decode.cu:
// mbarrier and bulk-copy PTX, the FP8 row codec in the page layout of
// include/mkv.h ("Storage formats"), and the TQ3 unit decoder (PRMT byte-table
// lookups of the fp16 levels).
#pragma once

#include "mkv_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace mkv {
namespace dev {

constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz: bound on any wait

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
// L2 policy for KV page data: read once per launch, it should not push the
// small, reused data (plan tables, q, partial states) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 1-D bulk copy global -> shared (16-byte aligned addresses and size), counted
// by an mbarrier's transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also returns the OR of a predicate over the threads.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
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

// ------------------------------------------------------------------ FP8 rows
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
// Byte offset of (token t, dim j) in an FP8 K / V plane's code bytes.  The
// offsets depend on t only through t % 64 and t / 64 (K) or t % 8 and t / 8
// (V), so a staged 64-token block uses them with t % 64.
__device__ __forceinline__ int fp8_k_off(int t, int j) {
  return (t >> 6) * (64 * kHeadDim) + (j >> 4) * 1024 + (t & 63) * 16 + (j & 15);
}
__device__ __forceinline__ int fp8_v_off(int t, int j) { return (t >> 3) * (8 * kHeadDim) + j * 8 + (t & 7); }
// Store a quantised row (lane's dims 8l .. 8l+7 in c) at token t of a K
// (kv = 0) or V (kv = 1) plane: codes at `codes`, fp16 scales at `scales`.
// Works on a page plane in global memory and on a staged 64-token block in
// shared memory alike (t < 64 there).
__device__ __forceinline__ void fp8_store_row(uint8_t* codes, uint8_t* scales, int kv, int t, int lane,
                                              const uint32_t (&c)[4], __half s16) {
  if (kv == 0) {
    uint2 w;
    w.x = c[0] | (c[1] << 16);
    w.y = c[2] | (c[3] << 16);
    *reinterpret_cast<uint2*>(codes + fp8_k_off(t, 8 * lane)) = w;
  } else {
    uint8_t* base = codes + fp8_v_off(t, 8 * lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      base[8 * (2 * i)] = static_cast<uint8_t>(c[i] & 0xff);
      base[8 * (2 * i + 1)] = static_cast<uint8_t>(c[i] >> 8);
    }
  }
  if (lane == 0) reinterpret_cast<__half*>(scales)[t] = s16;
}
// The 8 e4m3 bytes of row t (dims 8l .. 8l+7, l = lane) of a K / V plane.
__device__ __forceinline__ void fp8_load_row(const uint8_t* plane, int kv, int t, int lane, uint8_t (&b)[8]) {
  if (kv == 0) {
    const uint2 w = *reinterpret_cast<const uint2*>(plane + fp8_k_off(t, 8 * lane));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      b[i] = (w.x >> (8 * i)) & 0xff;
      b[4 + i] = (w.y >> (8 * i)) & 0xff;
    }
  } else {
    const uint8_t* r = plane + fp8_v_off(t, 8 * lane);
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = r[8 * i];
  }
}

// ------------------------------------------------------------------ TQ3 units
// Code e (0..31) of a 12-byte unit (words w0..w2).
__device__ __forceinline__ int tq3_unit_code(const uint32_t* w, int e) {
  if (e < 24) return (w[e >> 3] >> (4 * (e & 7))) & 7;
  const int i = e - 24;
  return ((w[0] >> (4 * i + 3)) & 1) | (((w[1] >> (4 * i + 3)) & 1) << 1) | (((w[2] >> (4 * i + 3)) & 1) << 2);
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
// Four 3-bit codes held as nibbles in sel[15:0] -> two f16x2 registers
// (codes 0,1) and (codes 2,3): PRMT looks the low and the high byte of each
// level up in 8-byte tables, then interleaves them.
__device__ __forceinline__ void tq3_lookup4(uint32_t sel, const Lut& t, uint32_t& h01, uint32_t& h23) {
  const uint32_t lo = __byte_perm(t.lo_a, t.lo_b, sel);
  const uint32_t hi = __byte_perm(t.hi_a, t.hi_b, sel);
  h01 = __byte_perm(lo, hi, 0x5140);
  h23 = __byte_perm(lo, hi, 0x7362);
}
// A unit's 32 codes as 16 f16x2 registers: r[i] = levels of codes 2i, 2i+1.
__device__ __forceinline__ void tq3_unit_levels(uint32_t w0, uint32_t w1, uint32_t w2, const Lut& lut, uint32_t* r) {
  uint32_t s[8];
  tq3_unit_selectors(w0, w1, w2, s);
#pragma unroll
  for (int k = 0; k < 8; ++k) tq3_lookup4(s[k], lut, r[2 * k], r[2 * k + 1]);
}

}  // namespace dev
}  // namespace mkv
