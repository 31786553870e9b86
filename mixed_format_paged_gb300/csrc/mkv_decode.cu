// Decode-attention kernel (sm_103a): partial attention states of FP8 and TQ3
// page runs on the fifth-generation tensor cores.
//
// Method: "Minima-KV: Retention-Preserving KV Cache Compression with
// Mixed-Format Paged Attention" (arXiv 2608.23834), abstract on the
// mlsanity.com paper page: "format-specific kernels compute partial attention
// states" (m, l, o) over Recent/Anchor FP8 pages and Stale TQ3 pages, which a
// globally normalised online-softmax merge (mkv_merge_kernel) combines.  TQ3
// pages are scored in the rotated domain: q' = R q is built once per piece
// and o' stays rotated until the merge applies R^T once.
//
// Structure.  One persistent CTA per SM, three warpgroups (WG) of 128 threads.
// The host cut the launch's tiles (128 tokens of TQ3, 64 tokens of FP8, of
// one (request, kv head, format) group) into one contiguous piece list per
// CTA; within a piece, WG w takes tiles w, w + 3, w + 6, ...  Each WG owns
//   - a ring of two shared-memory slots, filled by 1-D bulk copies issued by
//     its thread 0 and counted by one mbarrier per slot;
//   - 128 tensor-memory columns: A (64 columns: a dequantised K half or V
//     half, fp16 pairs), S (QK^T, 16 fp32 columns), O (P V, 2 x 16 fp32
//     columns, one per half of head_dim);
//   - a P' buffer in shared memory (the B operand of P V).
// Per tile, thread t of the WG (TMEM lane t):
//   K:  dequantises token t's K row half by half (TQ3: PRMT byte-table lookups
//       of the fp16 levels; FP8: cvt e4m3x2) and stores it to A with
//       tcgen05.st; thread 0 issues S += A q'^T (tcgen05.mma kind::f16, M 128,
//       N 16, K 16 per instruction; q' hi/lo fp16 rows in shared memory, so
//       S_hi + S_lo is fp32-accurate);
//   softmax: reads S row t (tcgen05.ld), scales by the token's K scale, and
//       forms p = 2^(s - m) against the WG's running max m (log2 units).  A
//       barrier with an OR-reduction flags scores more than 2^8 above m; then
//       (rarely) the WG takes the tile max, rescales O in tensor memory and
//       recomputes p.  P' = p * (V scale) goes to shared memory as fp16;
//   V:  dequantises head dimension t (and t + 128) across the tile's tokens
//       into A; thread 0 issues O_half += A P' (M 128 = dims, N 16 = heads,
//       K 16 = tokens per instruction).
// tcgen05.commit -> one mbarrier per WG tracks the MMAs; a thread never
// overwrites A or P' before the MMAs reading them completed.  At the end of a
// piece the three WGs' (m, l, O) merge, in a fixed order, into one partial
// state per q head.
//
// Every wait is bounded (about 2 s of SM clocks).  A wait that runs out sets
// a bit in the pool's device error word and the CTA's abort flag; the threads
// then keep passing the same barriers without waiting, so no thread is left
// behind at a barrier, and the CTA waits (bounded) for its copies and MMAs in
// flight before it frees its tensor memory and exits.
#include "mkv_device.cuh"

#include <atomic>

namespace mkv {
namespace {

using namespace dev;

constexpr int kWG = kDecWGs;                 // warpgroups per CTA
constexpr int kThreads = kWG * 128;
constexpr int kSlots = 2;                    // staging slots per WG
constexpr float kLazyRescale = 8.0f;         // log2 units a max may grow before O is rescaled
constexpr float kFp8PScale = 512.0f;         // keeps p * s in the fp16 normal range for FP8 V

// Slot layout of a TQ3 tile (128 tokens: two 64-token pages or one 128-token page)
constexpr int kT3K = 0;                      // K rows, token t at 96 t
constexpr int kT3V = 12288;                  // V: page j (64-token pages) at + 6144 j, dim d at + 24 d;
                                             //    one 128-token page: dim d at + 48 d
constexpr int kT3Ks = 24576;                 // K scales, token t at + 2 t
constexpr int kT3Vs = 24832;                 // V scales
constexpr int kT3Bytes = 25088;
// Slot layout of an FP8 tile (64 tokens: one 64-token block of a page)
constexpr int kF8K = 0;                      // K block (16 columns x 64 tokens x 16 B)
constexpr int kF8V = 16384;                  // V block (8 groups x 256 dims x 8 tokens)
constexpr int kF8Ks = 32768;
constexpr int kF8Vs = 32896;
constexpr int kF8Bytes = 33024;
constexpr int kSlotBytes = kF8Bytes;
static_assert(kT3Bytes <= kSlotBytes, "a TQ3 tile must fit a slot");

constexpr int kQBytes = 8192;                // q' B operand: 16 rows x 256 fp16
constexpr int kPBytes = 4096;                // P' B operand: 16 rows x 128 fp16
constexpr int kQSbo = 4096;                  // q': byte distance of rows 8..15 from rows 0..7
constexpr int kPSbo = 2048;                  // P': the same

// Tensor memory: 512 columns, WG w at 128 w
constexpr int kTmemCols = 512;
constexpr int kTA = 0, kTS = 64, kTO0 = 96, kTO1 = 112;

// Shared memory
constexpr int kSmRing = 0;
constexpr int kSmQ = kSmRing + kWG * kSlots * kSlotBytes;      // [2] q' buffers
constexpr int kSmP = kSmQ + 2 * kQBytes;                       // [kWG] P' buffers
constexpr int kSmRedM = kSmP + kWG * kPBytes;                  // [kWG][4 warps][kMaxGroup] floats
constexpr int kSmRedL = kSmRedM + kWG * 4 * kMaxGroup * 4;
constexpr int kSmStatM = kSmRedL + kWG * 4 * kMaxGroup * 4;    // [kWG][kMaxGroup] WG max
constexpr int kSmStatL = kSmStatM + kWG * kMaxGroup * 4;       // [kWG][kMaxGroup] WG sum
constexpr int kSmBars = kSmStatL + kWG * kMaxGroup * 4;        // full[kWG][kSlots], mma[kWG]
constexpr int kSmMisc = kSmBars + (kWG * kSlots + kWG) * 8;    // tmem base, abort flag
constexpr int kDecSmemBytes = kSmMisc + 16;
static_assert(kDecSmemBytes <= 227 * 1024, "decode shared memory exceeds the per-CTA limit");
static_assert(kSmQ % 16 == 0 && kSmP % 16 == 0 && kSmBars % 8 == 0, "operand buffers need 16-byte alignment");
static_assert(2 * kPBytes >= kHeadDim * kMaxGroup * 4 && kQBytes >= kHeadDim * kMaxGroup * 4,
              "the piece-end exchange reuses the P' and q' buffers");

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B fp16,
// both K-major, N = 16, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // canonical K-major layout without swizzle: 8-row x 16-byte core matrices,
  // lbo = distance of core matrices along K, sbo = along M/N; version 1
  return static_cast<uint64_t>((addr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(acc), "r"(kIdesc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ state
struct Smem {
  uint8_t* base;
  __device__ uint8_t* slot(int wg, int s) const { return base + kSmRing + (wg * kSlots + s) * kSlotBytes; }
  __device__ uint8_t* qbuf(int i) const { return base + kSmQ + i * kQBytes; }
  __device__ uint8_t* pbuf(int wg) const { return base + kSmP + wg * kPBytes; }
  __device__ float* red_m(int wg) const { return reinterpret_cast<float*>(base + kSmRedM) + wg * 4 * kMaxGroup; }
  __device__ float* red_l(int wg) const { return reinterpret_cast<float*>(base + kSmRedL) + wg * 4 * kMaxGroup; }
  __device__ float* stat_m() const { return reinterpret_cast<float*>(base + kSmStatM); }
  __device__ float* stat_l() const { return reinterpret_cast<float*>(base + kSmStatL); }
  __device__ uint64_t* full(int wg, int s) const { return reinterpret_cast<uint64_t*>(base + kSmBars) + wg * kSlots + s; }
  __device__ uint64_t* mma(int wg) const { return reinterpret_cast<uint64_t*>(base + kSmBars) + kWG * kSlots + wg; }
  __device__ uint32_t* tmem_base() const { return reinterpret_cast<uint32_t*>(base + kSmMisc); }
  __device__ int* abort_flag() const { return reinterpret_cast<int*>(base + kSmMisc + 4); }
};

__device__ __forceinline__ bool aborted(const Smem& sm) {
  return *reinterpret_cast<volatile int*>(sm.abort_flag()) != 0;
}
// Bounded wait; returns false at once when the CTA has aborted.
__device__ __forceinline__ bool dec_wait(const Smem& sm, uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (aborted(sm)) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(err, kErrWaitTimeout);
      *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
      return false;
    }
  }
}

struct Piece {                               // one CTA piece (its Segment)
  int fmt, b, kvh, entry0, nentry, tile0, ntile, part;
};
__device__ __forceinline__ Piece piece_of(const Segment& s) {
  return Piece{s.fmt, s.b, s.kvh, s.entry0, s.nentry, s.tile, s.ntile, s.part};
}
__device__ __forceinline__ Piece load_piece(const DecodeParams& p, int si) {
  return si == p.cta_seg[blockIdx.x] ? piece_of(p.first[blockIdx.x]) : piece_of(p.segs[si]);
}

// Tile k of a piece: its first page entry, the number of pages it spans (a
// TQ3 tile of 64-token pages spans two, unless the group ends), the first
// token within the page (FP8 tiles of 128-token pages take a half) and its
// valid tokens.
struct TileLoc {
  int e, npages, tok0, nv;
};
__device__ __forceinline__ TileLoc tile_locate(const DecodeParams& p, const Piece& pc, int k) {
  TileLoc t;
  const int kk = pc.tile0 + k;
  if (pc.fmt) {
    const int ppt = p.P == 64 ? 2 : 1;
    const int rel = kk * ppt;
    t.e = pc.entry0 + rel;
    t.npages = min(ppt, pc.nentry - rel);
    t.tok0 = 0;
    t.nv = t.npages * p.P;               // TQ3 pages are full
  } else {
    const int tpp = p.P / kFp8Tile;
    t.e = pc.entry0 + kk / tpp;
    t.npages = 1;
    t.tok0 = (kk % tpp) * kFp8Tile;
    t.nv = min(kFp8Tile, static_cast<int>(p.entries[t.e].nvalid) - t.tok0);
  }
  return t;
}

// Thread 0 of a WG: copy tile k of piece pc into slot st (mbarrier bar), or
// complete the slot's phase without bytes for an empty tile or a bad plan
// entry (an out-of-arena slot: reported, and the CTA aborts).
__device__ __noinline__ void dec_issue(const DecodeParams& p, const Piece& pc, int k, uint8_t* st, uint64_t* bar,
                                       int* abort_flag) {
  const TileLoc tl = tile_locate(p, pc, k);
  if (tl.nv <= 0) {
    mbar_arrive(bar);
    return;
  }
  const int nslots = pc.fmt ? p.tq3_slots : p.fp8_slots;
  for (int j = 0; j < tl.npages; ++j) {
    const int s = p.entries[tl.e + j].slot;
    if (s < 0 || s >= nslots) {
      atomicOr(p.err, kErrBadPlan);
      *reinterpret_cast<volatile int*>(abort_flag) = 1;
      mbar_arrive(bar);
      return;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const uint64_t pol = l2_evict_first_policy();
  if (pc.fmt) {
    const int codes = p.P * (3 * kHeadDim / 8), plane = codes + 2 * p.P;
    mbar_expect_tx(bar, tl.npages * 2 * plane);
    for (int j = 0; j < tl.npages; ++j) {
      const uint8_t* hp = p.tq3_layer + static_cast<int64_t>(p.entries[tl.e + j].slot) * p.tq3_page_bytes +
                          static_cast<int64_t>(pc.kvh) * 2 * plane;
      bulk_g2s(st + kT3K + j * codes, hp, codes, bar, pol);
      bulk_g2s(st + kT3Ks + j * 2 * p.P, hp + codes, 2 * p.P, bar, pol);
      bulk_g2s(st + kT3V + j * codes, hp + plane, codes, bar, pol);
      bulk_g2s(st + kT3Vs + j * 2 * p.P, hp + plane + codes, 2 * p.P, bar, pol);
    }
  } else {
    const int codes = p.P * kHeadDim, plane = codes + 2 * p.P;
    const int half = tl.tok0 / kFp8Tile;
    const uint8_t* hp = p.fp8_layer + static_cast<int64_t>(p.entries[tl.e].slot) * p.fp8_page_bytes +
                        static_cast<int64_t>(pc.kvh) * 2 * plane;
    mbar_expect_tx(bar, kF8Bytes);
    bulk_g2s(st + kF8K, hp + half * (kFp8Tile * kHeadDim), kFp8Tile * kHeadDim, bar, pol);
    bulk_g2s(st + kF8Ks, hp + codes + half * 2 * kFp8Tile, 2 * kFp8Tile, bar, pol);
    bulk_g2s(st + kF8V, hp + plane + half * (kFp8Tile * kHeadDim), kFp8Tile * kHeadDim, bar, pol);
    bulk_g2s(st + kF8Vs, hp + plane + codes + half * 2 * kFp8Tile, 2 * kFp8Tile, bar, pol);
  }
}

// The WG's sequence of tiles over the CTA's pieces (tile k of piece si,
// k = wg, wg + kWG, ...).  Every thread of the WG keeps the same cursor.
struct TileCursor {
  int si, s1, k;
  int issued;                                // tiles copied in so far (thread 0)
  Piece pc;
  __device__ void start(const DecodeParams& p, int s0, int s1_, int wg) {
    issued = 0;
    si = s0;
    s1 = s1_;
    k = wg;
    if (si < s1) pc = load_piece(p, si);
    settle(p, wg);
  }
  __device__ void settle(const DecodeParams& p, int wg) {
    while (si < s1 && k >= pc.ntile) {
      if (++si < s1) pc = load_piece(p, si);
      k = wg;
    }
  }
  __device__ bool valid() const { return si < s1; }
  __device__ void advance(const DecodeParams& p, int wg) {
    k += kWG;
    settle(p, wg);
  }
};

// ------------------------------------------------------------------ q'
// Raw q row h of piece pc (8 dims per lane: bf16 in r[0] or fp32 in r[0..1]);
// zeros for h >= G.  Loaded a piece ahead of its build.
struct QRow {
  uint4 r[2];
};
__device__ __forceinline__ QRow load_q_row(const DecodeParams& p, const Piece& pc, int h, int lane) {
  QRow q{};
  if (h < p.G) {
    const size_t off = (static_cast<size_t>(pc.b) * p.Hq + pc.kvh * p.G + h) * kHeadDim + 8 * lane;
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
// Row h of piece pc's B operand for QK^T, built by one warp from its raw q
// row: x = q (FP8 pieces) or q' = R q = (H D q) / 16 (TQ3 pieces; signs,
// then the Walsh-Hadamard butterflies, 8 dims per lane in registers and
// across lanes by shuffles).  Row h holds fp16(x), row 8 + h the fp16
// residual x - fp16(x).  Canonical K-major layout: element (n, k) at
// (k/8)*128 + (n/8)*kQSbo + (n%8)*16 + (k%8)*2, so lane l (dims 8l .. 8l+7)
// writes 16 bytes per row.
__device__ __forceinline__ void build_q_row(uint8_t* qb, const Piece& pc, int h, int lane, const QRow& q,
                                            uint32_t qsign, int q_bf16) {
  float x[8];
  if (q_bf16) {
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
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float h0 = __half2float(__float2half_rn(x[2 * i])), h1 = __half2float(__float2half_rn(x[2 * i + 1]));
    hi[i] = pack_half2(h0, h1);
    lo[i] = pack_half2(x[2 * i] - h0, x[2 * i + 1] - h1);
  }
  *reinterpret_cast<uint4*>(qb + lane * 128 + h * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(qb + lane * 128 + kQSbo + h * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// ------------------------------------------------------------------ dequantisation
// TQ3 K, half hf (dims 128 hf .. +127) of token t: four units, 64 f16x2
// registers (register i = dims 128 hf + 2i, +1).
__device__ __forceinline__ void deq_k_tq3(const uint8_t* st, int t, int hf, const Lut& lut, uint32_t (&r)[64]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(st + kT3K + t * 96 + hf * 48);
  const uint4 a = s4[0], b = s4[1], c = s4[2];
  tq3_unit_levels(a.x, a.y, a.z, lut, r);
  tq3_unit_levels(a.w, b.x, b.y, lut, r + 16);
  tq3_unit_levels(b.z, b.w, c.x, lut, r + 32);
  tq3_unit_levels(c.y, c.z, c.w, lut, r + 48);
}
// TQ3 V of head dimension d across the tile's 128 tokens (register i =
// tokens 2i, 2i+1): one 128-token page (four units at 48 d) or two 64-token
// pages (two units at 24 d each).
__device__ __forceinline__ void deq_v_tq3(const uint8_t* st, int d, int P, const Lut& lut, uint32_t (&r)[64]) {
  uint32_t w[12];
  if (P == 128) {
    const uint4* s4 = reinterpret_cast<const uint4*>(st + kT3V + d * 48);
    const uint4 a = s4[0], b = s4[1], c = s4[2];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y;
    w[6] = b.z; w[7] = b.w; w[8] = c.x; w[9] = c.y; w[10] = c.z; w[11] = c.w;
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint2* s2 = reinterpret_cast<const uint2*>(st + kT3V + j * 6144 + d * 24);
      const uint2 a = s2[0], b = s2[1], c = s2[2];
      w[6 * j + 0] = a.x; w[6 * j + 1] = a.y; w[6 * j + 2] = b.x;
      w[6 * j + 3] = b.y; w[6 * j + 4] = c.x; w[6 * j + 5] = c.y;
    }
  }
  tq3_unit_levels(w[0], w[1], w[2], lut, r);
  tq3_unit_levels(w[3], w[4], w[5], lut, r + 16);
  tq3_unit_levels(w[6], w[7], w[8], lut, r + 32);
  tq3_unit_levels(w[9], w[10], w[11], lut, r + 48);
}
// FP8 K, half hf of token t (t < 64): eight 16-byte columns.
__device__ __forceinline__ void deq_k_fp8(const uint8_t* st, int t, int hf, uint32_t (&r)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(st + kF8K + (8 * hf + c) * 1024 + t * 16);
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r[8 * c + 2 * i] = e4m3x2_to_f16x2(x[i]);
      r[8 * c + 2 * i + 1] = e4m3x2_to_f16x2(x[i] >> 16);
    }
  }
}
// FP8 V of head dimension d across the tile's 64 tokens: eight 8-token groups.
__device__ __forceinline__ void deq_v_fp8(const uint8_t* st, int d, uint32_t (&r)[64]) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint2 w = *reinterpret_cast<const uint2*>(st + kF8V + g * 2048 + d * 8);
    r[4 * g + 0] = e4m3x2_to_f16x2(w.x);
    r[4 * g + 1] = e4m3x2_to_f16x2(w.x >> 16);
    r[4 * g + 2] = e4m3x2_to_f16x2(w.y);
    r[4 * g + 3] = e4m3x2_to_f16x2(w.y >> 16);
  }
}

// Fused append (mkv_append_decode): warps 0 and 1 of the WG whose FP8 tile
// holds a request's newest token quantise the token's K and V rows and store
// them into the page (global memory, for later steps) and into the staged
// tile (whose copy predates them).
__device__ __forceinline__ void fused_append(const DecodeParams& p, const Piece& pc, const TileLoc& tl, uint8_t* st,
                                             int wwarp, int lane) {
  const PageEntry pe = p.entries[tl.e];
  const int pos = pe.nvalid - 1;
  if (!(pe.tail && pos >= tl.tok0 && pos < tl.tok0 + kFp8Tile) || wwarp > 1) return;
  if (pe.slot < 0 || pe.slot >= p.fp8_slots) return;   // a bad entry: dec_issue reported it
  const int kv = wwarp;
  const size_t row = (static_cast<size_t>(pc.b) * p.Hkv + pc.kvh) * kHeadDim;
  const int plane = p.P * (kHeadDim + 2);
  uint8_t* hp = p.fp8_layer + static_cast<int64_t>(pe.slot) * p.fp8_page_bytes +
                static_cast<int64_t>(pc.kvh) * 2 * plane + kv * plane;
  uint32_t c[4];
  __half s16;
  fp8_quantize_row(kv ? p.v : p.k, row, p.kv_bf16, lane, c, s16);
  fp8_store_row(hp, hp + p.P * kHeadDim, kv, pos, lane, c, s16);
  fp8_store_row(st + (kv ? kF8V : kF8K), st + (kv ? kF8Vs : kF8Ks), kv, pos - tl.tok0, lane, c, s16);
}

// ------------------------------------------------------------------ kernel
struct WgState {
  float m[kMaxGroup];          // running max per head (log2 units), the same in every thread of the WG
  float l[kMaxGroup];          // this thread's share of the running sum
  bool o_started;              // O holds this piece's sums
  uint32_t mma_cnt, mma_waited;
};

// Wait for the WG's latest MMA commit (if not yet waited for).
__device__ __forceinline__ void wait_mma(const DecodeParams& p, const Smem& sm, int wg, WgState& ws) {
  if (ws.mma_waited != ws.mma_cnt) {
    dec_wait(sm, sm.mma(wg), (ws.mma_cnt - 1) & 1, p.err);
    ws.mma_waited = ws.mma_cnt;
  }
  tc_fence_after();
}

// One tile of format FMT in slot st.
template <int FMT>
__device__ __forceinline__ void dec_tile(const DecodeParams& p, const Smem& sm, const Piece& pc, const TileLoc& tl,
                                         uint8_t* st, const uint8_t* qb, int wg, int wt, WgState& ws,
                                         uint32_t tbase) {
  const int wwarp = wt >> 5;
  const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * wwarp) << 16);   // this warp's TMEM lanes
  const uint32_t colA = tbase + kTA, colS = tbase + kTS;
  const int bar_id = 1 + wg;
  const bool issuer = wt == 0;
  const Lut& lut = p.lut;
  uint32_t r[64];
  uint8_t* pb = sm.pbuf(wg);
  // ---------------- S = K q'^T, two halves of head_dim
#pragma unroll 1
  for (int hf = 0; hf < 2; ++hf) {
    const bool rows = FMT == 1 || wt < kFp8Tile;      // FP8 tiles fill TMEM lanes 0..63
    if (FMT == 1)
      deq_k_tq3(st, wt, hf, lut, r);
    else if (rows)
      deq_k_fp8(st, wt, hf, r);
    wait_mma(p, sm, wg, ws);                          // A is free
    if (FMT == 1 || wwarp < 2) {
      tmem_st32(lane_base + kTA, r);
      tmem_st32(lane_base + kTA + 32, r + 32);
    }
    tmem_wait_st();
    tc_fence_before();
    named_bar(bar_id, 128);
    if (issuer) {
      tc_fence_after();
      const uint32_t qa = smem_addr(qb);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        mma_f16_tmem_a(colS, colA + 8 * j, smem_desc(qa + (8 * hf + j) * 256, 128, kQSbo), hf | j);
      mma_commit(sm.mma(wg));
    }
    ++ws.mma_cnt;
  }
  // ---------------- V half 0 into registers while QK runs
  if (FMT == 1)
    deq_v_tq3(st, wt, p.P, lut, r);
  else
    deq_v_fp8(st, wt, r);
  wait_mma(p, sm, wg, ws);                            // S is ready, A is free
  float sv[16];
  tmem_ld16(lane_base + kTS, sv);
  const int G = p.G;
  const bool valid = wt < tl.nv;
  const float ks = valid ? __half2float(reinterpret_cast<const __half*>(st + (FMT ? kT3Ks : kF8Ks))[wt]) : 0.f;
  const float vs = valid ? __half2float(reinterpret_cast<const __half*>(st + (FMT ? kT3Vs : kF8Vs))[wt]) *
                               (FMT ? 1.f : kFp8PScale)
                         : 0.f;
  float s[kMaxGroup];
  bool need = false;
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    s[h] = (valid && h < G) ? (sv[h] + sv[8 + h]) * (ks * p.score_scale) : -INFINITY;
    need |= s[h] > ws.m[h] + kLazyRescale;
  }
  // p = 2^(s - m) and P' = p * (V scale), against the current max (a max of
  // -inf, for a head with no score yet, is taken as 0: every score is then
  // -inf too and p = 0)
  float pr[kMaxGroup];
  auto write_p = [&]() {
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h < G) {
        pr[h] = ex2(s[h] - (ws.m[h] == -INFINITY ? 0.f : ws.m[h]));
        *reinterpret_cast<__half*>(pb + (wt >> 3) * 128 + h * 16 + (wt & 7) * 2) = __float2half_rn(pr[h] * vs);
      }
    }
  };
  write_p();
  tmem_st32(lane_base + kTA, r);
  if (FMT == 1) tmem_st32(lane_base + kTA + 32, r + 32);
  tmem_wait_st();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  if (named_bar_or(bar_id, 128, need)) {
    // a score grew past the lazy bound: move the max to the tile's max
    float* rm = sm.red_m(wg);
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      float x = s[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
      if ((wt & 31) == 0) rm[wwarp * kMaxGroup + h] = x;
    }
    named_bar(bar_id, 128);
    float alpha[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      const float tm = fmaxf(fmaxf(rm[h], rm[kMaxGroup + h]), fmaxf(rm[2 * kMaxGroup + h], rm[3 * kMaxGroup + h]));
      const float mn = fmaxf(ws.m[h], tm);
      alpha[h] = (ws.m[h] == -INFINITY) ? 0.f : ex2(ws.m[h] - mn);
      ws.m[h] = mn;
      ws.l[h] *= alpha[h];
    }
    if (ws.o_started) {
      float o[16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t col = lane_base + (c ? kTO1 : kTO0);
        tmem_ld16(col, o);
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) o[h] *= alpha[h];
        tmem_st16f(col, o);
      }
      tmem_wait_st();
    }
    write_p();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    named_bar(bar_id, 128);          // also keeps red_m live until every thread read it
  }
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h)
    if (h < G) ws.l[h] += pr[h];
  const int nj = FMT == 1 ? 8 : 4;                    // 16-token K steps of P V
  if (issuer) {
    tc_fence_after();
    const uint32_t pa = smem_addr(pb);
    for (int j = 0; j < nj; ++j)
      mma_f16_tmem_a(tbase + kTO0, colA + 8 * j, smem_desc(pa + j * 256, 128, kPSbo), (ws.o_started || j) ? 1u : 0u);
    mma_commit(sm.mma(wg));
  }
  ++ws.mma_cnt;
  // ---------------- V half 1
  if (FMT == 1)
    deq_v_tq3(st, 128 + wt, p.P, lut, r);
  else
    deq_v_fp8(st, 128 + wt, r);
  wait_mma(p, sm, wg, ws);
  tmem_st32(lane_base + kTA, r);
  if (FMT == 1) tmem_st32(lane_base + kTA + 32, r + 32);
  tmem_wait_st();
  tc_fence_before();
  named_bar(bar_id, 128);                              // the slot is no longer read
  if (issuer) {
    tc_fence_after();
    const uint32_t pa = smem_addr(pb);
    for (int j = 0; j < nj; ++j)
      mma_f16_tmem_a(tbase + kTO1, colA + 8 * j, smem_desc(pa + j * 256, 128, kPSbo), (ws.o_started || j) ? 1u : 0u);
    mma_commit(sm.mma(wg));
  }
  ++ws.mma_cnt;
  ws.o_started = true;
}

// End of a piece: the three WGs' states merge into the piece's partial state.
// Each WG's O is scaled to the common max of each head; WGs 1 and 2 hand
// theirs over through shared memory (the P' buffers and this piece's q'
// buffer, free once every MMA of the piece completed) and WG 0 adds them in a
// fixed order and writes (m, l, o) per q head.
__device__ __forceinline__ void dec_piece_end(const DecodeParams& p, const Smem& sm, const Piece& pc, int pi, int wg,
                                              int wt, WgState& ws, uint32_t tbase) {
  const int G = p.G, wwarp = wt >> 5, lane = wt & 31;
  wait_mma(p, sm, wg, ws);
  float* rl = sm.red_l(wg);
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    float x = ws.l[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    if (lane == 0) rl[wwarp * kMaxGroup + h] = x;
  }
  named_bar(1 + wg, 128);
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h)
    if (wt == h) {
      sm.stat_m()[wg * kMaxGroup + h] = ws.m[h];
      sm.stat_l()[wg * kMaxGroup + h] = ((rl[h] + rl[kMaxGroup + h]) + rl[2 * kMaxGroup + h]) + rl[3 * kMaxGroup + h];
    }
  __syncthreads();
  float f[kMaxGroup];
  const float osc = pc.fmt ? 1.f : 1.f / kFp8PScale;
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWG; ++w) M = fmaxf(M, sm.stat_m()[w * kMaxGroup + h]);
    f[h] = (ws.m[h] == -INFINITY) ? 0.f : ex2(ws.m[h] - M) * osc;
  }
  float o0[16], o1[16];
  const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * wwarp) << 16);
  if (ws.o_started) {
    tmem_ld16(lane_base + kTO0, o0);
    tmem_ld16(lane_base + kTO1, o1);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) o0[i] = o1[i] = 0.f;
  }
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    o0[h] = f[h] == 0.f ? 0.f : o0[h] * f[h];
    o1[h] = f[h] == 0.f ? 0.f : o1[h] * f[h];
  }
  // exchange buffers [256 dims][kMaxGroup] floats
  float* xb = wg == 1 ? reinterpret_cast<float*>(sm.pbuf(0)) : reinterpret_cast<float*>(sm.qbuf(pi & 1));
  if (wg > 0) {
    float4* a = reinterpret_cast<float4*>(xb + wt * kMaxGroup);
    float4* b = reinterpret_cast<float4*>(xb + (128 + wt) * kMaxGroup);
    a[0] = make_float4(o0[0], o0[1], o0[2], o0[3]);
    a[1] = make_float4(o0[4], o0[5], o0[6], o0[7]);
    b[0] = make_float4(o1[0], o1[1], o1[2], o1[3]);
    b[1] = make_float4(o1[4], o1[5], o1[6], o1[7]);
  }
  __syncthreads();
  if (wg == 0) {
    const float* x1 = reinterpret_cast<const float*>(sm.pbuf(0));
    const float* x2 = reinterpret_cast<const float*>(sm.qbuf(pi & 1));
    float* dst = p.part + static_cast<size_t>(pc.part) * G * (2 + kHeadDim);
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h < G) {
        dst[h * (2 + kHeadDim) + 2 + wt] = (o0[h] + x1[wt * kMaxGroup + h]) + x2[wt * kMaxGroup + h];
        dst[h * (2 + kHeadDim) + 2 + 128 + wt] =
            (o1[h] + x1[(128 + wt) * kMaxGroup + h]) + x2[(128 + wt) * kMaxGroup + h];
      }
    }
    if (wt < G) {
      float M = -INFINITY, L = 0.f;
#pragma unroll
      for (int w = 0; w < kWG; ++w) M = fmaxf(M, sm.stat_m()[w * kMaxGroup + wt]);
#pragma unroll
      for (int w = 0; w < kWG; ++w) {
        const float mw = sm.stat_m()[w * kMaxGroup + wt];
        if (mw != -INFINITY) L += ex2(mw - M) * sm.stat_l()[w * kMaxGroup + wt];
      }
      dst[wt * (2 + kHeadDim)] = M;
      dst[wt * (2 + kHeadDim) + 1] = L;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) mkv_decode_kernel(DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem sm{smem_raw};
  const int s0 = p.cta_seg[blockIdx.x], s1 = p.cta_seg[blockIdx.x + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7, wt = tid & 127;
  // the merge kernel that follows waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t qsign = static_cast<uint32_t>(
      (lane < 8 ? p.signs[0] : lane < 16 ? p.signs[1] : lane < 24 ? p.signs[2] : p.signs[3]) >> (8 * (lane & 7))) & 0xFFu;
  if (tid == 0) {
    for (int w = 0; w < kWG; ++w) {
      for (int s = 0; s < kSlots; ++s) mbar_init(sm.full(w, s), 1);
      mbar_init(sm.mma(w), 1);
    }
    *sm.abort_flag() = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(sm.tmem_base())),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *sm.tmem_base() + 128 * wg;
  // q, the KV pages (demotion) and the partial-state workspace belong to the
  // preceding kernels: wait for them first
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool q_warp = warp < p.G;
  TileCursor ic;
  ic.start(p, s0, s1, wg);
  if (wt == 0) {
    for (int s = 0; s < kSlots && ic.valid(); ++s) {
      dec_issue(p, ic.pc, ic.k, sm.slot(wg, s), sm.full(wg, s), sm.abort_flag());
      ++ic.issued;
      ic.advance(p, wg);
    }
  } else {
    for (int s = 0; s < kSlots && ic.valid(); ++s) ic.advance(p, wg);
  }
  if (q_warp && s0 < s1) build_q_row(sm.qbuf(0), load_piece(p, s0), warp, lane, load_q_row(p, load_piece(p, s0), warp, lane),
                                     qsign, p.q_bf16);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  WgState ws;
  ws.mma_cnt = ws.mma_waited = 0;
  int slot = 0;
  uint32_t phase = 0;
  for (int si = s0; si < s1; ++si) {
    const int pi = si - s0;
    const Piece pc = load_piece(p, si);
    const bool prep_next = si + 1 < s1 && q_warp;
    Piece pn{};
    QRow qn{};
    if (prep_next) {
      pn = load_piece(p, si + 1);
      qn = load_q_row(p, pn, warp, lane);
    }
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      ws.m[h] = -INFINITY;
      ws.l[h] = 0.f;
    }
    ws.o_started = false;
    const uint8_t* qb = sm.qbuf(pi & 1);
    for (int k = wg; k < pc.ntile; k += kWG) {
      const TileLoc tl = tile_locate(p, pc, k);
      dec_wait(sm, sm.full(wg, slot), phase, p.err);
      uint8_t* st = sm.slot(wg, slot);
      if (pc.fmt == 0 && p.append) {
        fused_append(p, pc, tl, st, wt >> 5, lane);
        named_bar(1 + wg, 128);
      }
      if (pc.fmt)
        dec_tile<1>(p, sm, pc, tl, st, qb, wg, wt, ws, tbase);
      else
        dec_tile<0>(p, sm, pc, tl, st, qb, wg, wt, ws, tbase);
      // the slot is free (every thread passed the last barrier of the tile):
      // copy in the WG's tile kSlots further on
      if (ic.valid()) {
        if (wt == 0 && !aborted(sm)) {
          dec_issue(p, ic.pc, ic.k, st, sm.full(wg, slot), sm.abort_flag());
          ++ic.issued;
        }
        ic.advance(p, wg);
      }
      if (++slot == kSlots) {
        slot = 0;
        phase ^= 1;
      }
    }
    dec_piece_end(p, sm, pc, pi, wg, wt, ws, tbase);
    if (si + 1 < s1) {
      if (prep_next) build_q_row(sm.qbuf((pi + 1) & 1), pn, warp, lane, qn, qsign, p.q_bf16);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
    }
  }
  // on the normal path every copy and MMA was waited for; after an abort,
  // wait (bounded) for those still in flight before the CTA frees its tensor
  // memory and exits
  __syncthreads();
  if (aborted(sm) && wt == 0) {
    for (int j = ic.issued > kSlots ? ic.issued - kSlots : 0; j < ic.issued; ++j) {
      const long long t0 = clock64();
      while (!mbar_try_wait(sm.full(wg, j % kSlots), (j / kSlots) & 1))
        if (clock64() - t0 > kWaitCycles) break;
    }
    if (ws.mma_cnt != 0) {
      const long long t0 = clock64();
      while (!mbar_try_wait(sm.mma(wg), (ws.mma_cnt - 1) & 1))
        if (clock64() - t0 > kWaitCycles) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*sm.tmem_base()), "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

size_t decode_smem_bytes() { return kDecSmemBytes; }
int decode_threads() { return kThreads; }

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
  // the shared-memory limit is a per-device attribute: set it once per device
  // (setting it twice from racing threads is harmless)
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(mkv_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_acq_rel);
  }
  if (p.n_ctas <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDecSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mkv_decode_kernel, p);
}

}  // namespace mkv
