// CUDA kernels (sm_103a) of the mixed-format paged decode-attention library,
// other than the decode kernel itself (mkv_decode.cu).
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
//   mkv_dequant_kernel -- dense export of pages (FP8 or TQ3, rotated back)
//   mkv_merge_kernel   -- LSE merge: TQ3 partials in the rotated domain,
//                         one R^T, then FP8 partials; writes out and lse
#include "mkv_device.cuh"

namespace mkv {
namespace {

using namespace dev;

// ============================================================== append
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
  fp8_store_row(plane, plane + P * kHeadDim, kv, pos, lane, c, s16);
}

// ============================================================== demote
// One block per (page pair, layer, kv head, K|V plane).  Each warp encodes
// rows (dequantise, sign flip, 8-stage FWHT, RMS scale, threshold count);
// the block then packs 12-byte units (K token-major, V dimension-major) and
// writes the TQ3 plane.
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
    fp8_load_row(src, kv, t, lane, b);
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
  // pack units: word w -> unit w/3, word index k = w%3; unit u holds
  // K: token u/(d/32), dims 32*(u%(d/32)) + e;  V: dim u/(P/32), tokens 32*(u%(P/32)) + e
  const int nwords = P * (kHeadDim / 32) * 3;
  uint32_t* out = reinterpret_cast<uint32_t*>(dst);
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) {
    const int unit = w / 3, k = w - 3 * (w / 3);
    int t0, j0, dt, dj;
    if (kv == 0) {
      t0 = unit / (kHeadDim / 32);
      j0 = (unit % (kHeadDim / 32)) * 32;
      dt = 0;
      dj = 1;
    } else {
      j0 = unit / (P / 32);
      t0 = (unit % (P / 32)) * 32;
      dt = 1;
      dj = 0;
    }
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e0 = 8 * k + i, e1 = 24 + i;
      const uint32_t c0 = codes[(t0 + dt * e0) * kHeadDim + j0 + dj * e0];
      const uint32_t c1 = codes[(t0 + dt * e1) * kHeadDim + j0 + dj * e1];
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
    fp8_load_row(base, kv, t, lane, b);
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
        unit = j * (P / 32) + t / 32;
        e = t % 32;
      }
      const uint32_t* w = reinterpret_cast<const uint32_t*>(base + 12 * unit);
      x[i] = sg * p.level[tq3_unit_code(w, e)];
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

// ============================================================== merge
// One block (256 threads, thread = dim) per (request, kv head, q head).  Each
// format's partial states merge in one pass with a running (M, L, O) -- the
// online-softmax recurrence, in partial-state order, so the result does not
// depend on timing -- loading eight partials at a time.  The TQ3 partials
// merge in the rotated domain, R^T is applied once (FWHT across the block,
// then the signs and 1/16), the FP8 partials join, and out = O / L,
// lse = (M + log2 L) ln 2.
constexpr int kMergeBatch = 8;

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
// batch is passed in already loaded.
__device__ __forceinline__ void merge_run(const float* part, int stride, int h, int first, int count, int d,
                                          const MergeBatch& first_batch, float& M, float& L, float& O) {
  M = -INFINITY;
  L = 0.f;
  O = 0.f;
  merge_fold(first_batch, M, L, O);
  for (int base = kMergeBatch; base < count; base += kMergeBatch) {
    MergeBatch mb;
    merge_load(part, stride, h, first, base, count, d, mb);
    merge_fold(mb, M, L, O);
  }
}

__global__ void __launch_bounds__(256) mkv_merge_kernel(MergeParams p) {
  __shared__ float xs[kHeadDim];
  const int h = blockIdx.x % p.G;
  const int bk = blockIdx.x / p.G;
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  // the merge descriptors come with the plan (copied in before the decode
  // kernel started), so they load while the decode kernel still runs
  const MergeDesc md = p.desc[bk];
  const bool neg = sign_neg(p.signs, threadIdx.x);
  // launched as a programmatic dependent of the decode kernel: wait for its
  // partial states before reading them
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int d = threadIdx.x, lane = d & 31;
  const int stride = p.G * (2 + kHeadDim);
  // the first batch of both formats goes out at once
  MergeBatch bs, bf;
  merge_load(p.part, stride, h, md.tq3_first, 0, md.tq3_count, d, bs);
  merge_load(p.part, stride, h, md.fp8_first, 0, md.fp8_count, d, bf);
  float Ms, Ls, os, Mf, Lf, of;
  merge_run(p.part, stride, h, md.tq3_first, md.tq3_count, d, bs, Ms, Ls, os);
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
  merge_run(p.part, stride, h, md.fp8_first, md.fp8_count, d, bf, Mf, Lf, of);
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

cudaError_t launch_dequant(const DequantParams& p, cudaStream_t s) {
  const int rows = p.npages * p.P * p.Hkv * 2;
  if (rows > 0) mkv_dequant_kernel<<<(rows + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
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
