// Internal structures shared by the host pool (mkv_host.cpp) and the CUDA
// kernels (mkv_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace mkv {

constexpr int kHeadDim = 256;      // head_dim the kernels are written for
constexpr int kMaxGroup = 8;       // q heads per kv head held in one MMA tile
constexpr int kDecWarps = 12;     // warps of a decode CTA (a piece's blocks go round-robin)
constexpr int kDecWarpsPair = 8;  // warps of a decode CTA whose batch entries hold two query tokens
// warps of a decode CTA with `qpe` query tokens per batch entry
constexpr int dec_warps(int qpe) { return qpe == 1 ? kDecWarps : kDecWarpsPair; }
constexpr int kFp8Blk = 16;        // tokens per FP8 decode block (one MMA tile)
constexpr int kTq3Blk = 32;        // tokens per TQ3 decode block (two MMA tiles)
constexpr int kTileTokens = 16;    // tokens per consumer-warp tile
constexpr int kMaxCtas = 160;      // upper bound on decode CTAs (their plan heads travel as kernel parameters)
constexpr int kQfragWords = 2048;  // A-fragment words of one piece's q rows (16 x 256 fp16)

// Error bits written by kernels into the pool's device error word.
enum : int {
  kErrWaitTimeout = 1,     // a bounded mbarrier wait ran out
  kErrBadPlan = 2,         // a plan entry pointed outside the arena
};

struct PageEntry {         // one page of one batch entry in a decode plan
  int32_t slot;            // physical slot in the tier's arena
  int16_t nvalid;          // tokens written in the page (1..P)
  int16_t tail;            // 1 for a request's last page: it may be written by the
                           // kernel just before the decode kernel (fused append);
                           // kTailPairLast for the last page of a paired entry
                           // whose first query token does not see the last token
};
constexpr int16_t kTailPairLast = 2;

struct Group {             // one run of pages: (request, kv head, format)
  int32_t b;               // batch index
  int32_t kvh;             // kv head
  int32_t fmt;             // 0 = FP8 (Recent/Anchor), 1 = TQ3 (Stale)
  int32_t entry0;          // first PageEntry
  int32_t nentry;          // number of PageEntry
  int32_t part0;           // first partial-state index of the group
  int32_t nparts;          // partial states (CTA pieces) of the group
  int32_t tokens;          // valid tokens (host bookkeeping)
};

struct Segment {           // one CTA's piece of one group: all the decode kernel reads about it
  int32_t fmt;             // 0 = FP8 (Recent/Anchor), 1 = TQ3 (Stale)
  int32_t b;               // batch index
  int32_t kvh;             // kv head
  int32_t entry0;          // the group's first PageEntry
  int32_t blk;             // first block of the piece, counted within the group:
                           // block k covers tokens [bt (k % bpp), +bt) of page
                           // entry0 + k / bpp (bt = kFp8Blk or kTq3Blk, bpp = P / bt)
  int32_t nblk;            // blocks in the piece
  int32_t part;            // partial-state index the piece writes
  int32_t group;           // the group (host bookkeeping)
};

struct MergeDesc {         // partial-state index ranges of one (b, kvh)
  int32_t tq3_first, tq3_count, fp8_first, fp8_count;
};

struct Codebook {          // stored TQ3 codebook (library constant)
  float level[8];          // fp16-valued levels, ascending
  float thr[7];            // thresholds (exact midpoints)
  uint16_t level_bits[8];  // fp16 bit patterns of the levels
};

struct Lut {               // byte tables for the PRMT level lookup
  uint32_t lo_a, lo_b, hi_a, hi_b;
};

struct DecodeParams {
  // scalars first, so that the kernel's first parameter loads bring them in together
  uint8_t* fp8_layer;              // FP8 arena base of this layer (written by the fused append)
  const uint8_t* tq3_layer;        // TQ3 arena base of this layer
  int64_t fp8_page_bytes, tq3_page_bytes;
  const PageEntry* entries;
  const Group* groups;
  const Segment* segs;             // per-CTA pieces, CTA by CTA
  const void* q;                   // [n, Hq, D], fp32 or bf16
  float* part;                     // [parts][qpe * G][2 + D] (m in log2 units, l, o)
  // fused single-token append (mkv_append_decode): each request's newest
  // token (the last valid one of its tail page), rows k/v [n, Hkv, D]
  const void* k;
  const void* v;
  int* err;
  uint64_t signs[4];               // rotation signs (bit i set: negative)
  Lut lut;
  int32_t fp8_slots, tq3_slots;
  int32_t n_ctas;
  int32_t q_bf16;
  int32_t Hq, Hkv, G, P;
  float score_scale;               // log2(e) / sqrt(d)
  int32_t append;
  int32_t kv_bf16;
  // query tokens: batch entry b holds query tokens s < qpe (1, or 2 for the
  // paired multi-query decode); its q / out row is q_row(b, s) (see below)
  int32_t qpe, nq, npair;
  // per CTA: when `heads` is set (graph launches), CTA i's pieces are
  // segs[heads[i] .. heads[i + 1]) and cta_seg / first are unused
  const int32_t* heads;
  int32_t cta_seg[kMaxCtas + 1];   // CTA i's pieces: segs[cta_seg[i] .. cta_seg[i + 1])
  Segment first[kMaxCtas];         // each CTA's first piece (a copy of segs[cta_seg[i]])
};

struct MergeParams {
  const float* part;
  const MergeDesc* desc;           // [n * Hkv]
  float* out;                      // [rows, Hq, D]
  float* lse;                      // [rows, Hq]
  int32_t n, Hq, Hkv, G;
  int32_t qpe, nq, npair;          // as in DecodeParams
  uint64_t signs[4];
};

// Row of q / out / lse for query token s of batch entry b.  One query token
// per entry (qpe 1): row b.  Paired entries (qpe 2; nq query tokens per
// request, npair = ceil(nq / 2) entries per request): entry b is request
// b / npair with its query tokens 2 (b % npair) and 2 (b % npair) + 1; with
// nq odd the last entry's second token repeats its first.
__host__ __device__ inline int q_row(int b, int s, int qpe, int nq, int npair) {
  if (qpe == 1) return b;
  const int r = b / npair, j = b - r * npair;
  const int i = 2 * j + s;
  return r * nq + (i < nq ? i : nq - 1);
}

struct AppendParams {
  uint8_t* fp8_layer;              // FP8 arena base of this layer
  int64_t fp8_page_bytes;
  const uint32_t* dest;            // per token: (slot << 8) | position in page
  const void* k;                   // [ntok, Hkv, D]
  const void* v;
  int32_t kv_bf16;
  int32_t ntok, Hkv, P;
};

struct DemoteParams {
  const uint8_t* fp8_arena;
  uint8_t* tq3_arena;
  int64_t fp8_page_bytes, tq3_page_bytes;
  int64_t fp8_layer_stride, tq3_layer_stride;   // bytes between layers
  const int2* pairs;               // (fp8 slot, tq3 slot)
  int32_t npairs, L, Hkv, P;
  uint64_t signs[4];
  float thr[7];
};

struct DequantParams {
  const uint8_t* fp8_layer;
  const uint8_t* tq3_layer;
  int64_t fp8_page_bytes, tq3_page_bytes;
  const int2* pages;               // (slot, tier << 16 | valid tokens) per page
  int32_t npages, Hkv, P;
  int32_t out_bf16;
  void* k_out;                     // [npages * P, Hkv, D]
  void* v_out;
  uint64_t signs[4];
  float level[8];
};

struct RelevanceParams {
  const uint8_t* fp8_layer;
  const uint8_t* tq3_layer;
  int64_t fp8_page_bytes, tq3_page_bytes;
  const int4* pages;               // per CTA: (batch index, page index, slot, tier << 16 | valid tokens)
  int32_t npages, Hq, Hkv, G, P;
  const void* q;                   // [n, Hq, D]
  int32_t q_bf16;
  const float* lse;                // [n, Hq], natural log over q . k / sqrt(D)
  float* mass;                     // [n, mass_stride]
  int32_t mass_stride;
  uint64_t signs[4];
  float level[8];
};

// Kernel launchers (mkv_kernels.cu).  Return cudaGetLastError() of the launch.
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_demote(const DemoteParams& p, cudaStream_t s);
// Launched with programmatic stream serialisation: its first page copies start
// while the preceding kernel finishes; it waits for that kernel before reading
// q or writing partial states.
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s);
// Sets the decode and merge kernels' per-device launch attributes (done by
// launch_decode too); call it before capturing decode launches into a graph.
cudaError_t prepare_decode_launch();
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);
cudaError_t launch_dequant(const DequantParams& p, cudaStream_t s);
cudaError_t launch_relevance(const RelevanceParams& p, cudaStream_t s);
size_t decode_smem_bytes();
// Device address and size of the library's fixed partial-state scratch (see
// mkv_decode_attention_noalloc), looked up for the current device on every
// call.
cudaError_t noalloc_scratch(float** ptr, size_t* bytes);
int decode_threads();

}  // namespace mkv
