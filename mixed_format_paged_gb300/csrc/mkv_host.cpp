// Host side of the mixed-format paged decode-attention library: page pool,
// page table and tier tags, free lists, decode planning, uploads and the C
// ABI declared in include/mkv.h.
//
// Method: "Minima-KV: Retention-Preserving KV Cache Compression with
// Mixed-Format Paged Attention" (arXiv 2608.23834), abstract (mlsanity.com):
// Recent and protected Anchor pages in FP8, older non-anchor pages in packed
// TQ3, every live-request page addressable; the setupai.cc summary
// ("Technical Deep Dive") places the formats in PagedAttention's block
// structure.  Everything here is bookkeeping; all arithmetic on cache data
// runs in mkv_kernels.cu.
#include "mkv.h"
#include "mkv_internal.h"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cstddef>
#include <functional>
#include <new>
#include <queue>
#include <string>
#include <utility>
#include <vector>

namespace mkv {
// mkv_selftest.cu: one CTA waits (bounded) on an mbarrier nothing arrives on
cudaError_t launch_wait_probe(int* err, long long limit_cycles, cudaStream_t s);
}  // namespace mkv

namespace {

using namespace mkv;

thread_local std::string g_last_error = "no error";

mkv_status fail(mkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ------------------------------------------------------------------ codebook
// 8-level Lloyd-Max quantiser for N(0,1) (Lloyd's alternation: thresholds at
// midpoints, levels at cell centroids), levels rounded to fp16.  Written from
// the mathematics; independent of any other implementation in the repository.
double phi(double x) { return std::isfinite(x) ? std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI) : 0.0; }
double Phi(double x) {
  if (x == INFINITY) return 1.0;
  if (x == -INFINITY) return 0.0;
  return 0.5 * std::erfc(-x / std::sqrt(2.0));
}

// IEEE binary16 round-to-nearest-even of a double; returns the value and bits.
double round_fp16(double v, uint16_t* bits) {
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (a == 0.0) {
    *bits = sign;
    return v;
  }
  int e;
  std::frexp(a, &e);          // a = f * 2^e, f in [0.5, 1)
  int ex = std::max(e - 1, -14);
  const double q = std::ldexp(1.0, ex - 10);
  double r = std::nearbyint(a / q) * q;   // default rounding mode: ties to even
  if (r > 65504.0) {
    *bits = sign | 0x7C00;
    return std::copysign(INFINITY, v);
  }
  // encode
  uint16_t b;
  if (r < std::ldexp(1.0, -14)) {
    b = static_cast<uint16_t>(std::nearbyint(r / std::ldexp(1.0, -24)));
  } else {
    int er;
    const double f = std::frexp(r, &er);   // r = f 2^er
    const int E = er - 1;                  // r in [2^E, 2^(E+1))
    const int man = static_cast<int>(std::nearbyint((f * 2.0 - 1.0) * 1024.0));
    b = static_cast<uint16_t>(((E + 15) << 10) | man);
  }
  *bits = sign | b;
  return std::copysign(r, v);
}

Codebook make_codebook() {
  double lv[8];
  for (int k = 0; k < 8; ++k) lv[k] = -2.0 + 4.0 * k / 7.0;
  for (int it = 0; it < 10000; ++it) {
    double edge[9];
    edge[0] = -INFINITY;
    edge[8] = INFINITY;
    for (int k = 1; k < 8; ++k) edge[k] = 0.5 * (lv[k - 1] + lv[k]);
    double delta = 0.0;
    for (int k = 0; k < 8; ++k) {
      const double c = (phi(edge[k]) - phi(edge[k + 1])) / (Phi(edge[k + 1]) - Phi(edge[k]));
      delta = std::max(delta, std::fabs(c - lv[k]));
      lv[k] = c;
    }
    if (delta < 1e-15) break;
  }
  Codebook cb;
  for (int k = 0; k < 8; ++k) cb.level[k] = static_cast<float>(round_fp16(lv[k], &cb.level_bits[k]));
  for (int k = 1; k < 8; ++k) cb.thr[k - 1] = static_cast<float>(0.5 * (double(cb.level[k - 1]) + cb.level[k]));
  return cb;
}

const Codebook& codebook() {
  static const Codebook cb = make_codebook();
  return cb;
}

Lut make_lut(const Codebook& cb) {
  Lut t{};
  for (int k = 0; k < 4; ++k) {
    t.lo_a |= uint32_t(cb.level_bits[k] & 0xff) << (8 * k);
    t.lo_b |= uint32_t(cb.level_bits[k + 4] & 0xff) << (8 * k);
    t.hi_a |= uint32_t(cb.level_bits[k] >> 8) << (8 * k);
    t.hi_b |= uint32_t(cb.level_bits[k + 4] >> 8) << (8 * k);
  }
  return t;
}

// ------------------------------------------------------------------ SplitMix64
// Steele, Lea, Flood, "Fast splittable pseudorandom number generators"
// (OOPSLA 2014): state advances by the golden gamma, output is the state
// mixed by two xor-shift-multiply rounds and a final xor-shift.
uint64_t splitmix64_next(uint64_t& state) {
  state += 0x9E3779B97F4A7C15ull;
  uint64_t z = state;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// ------------------------------------------------------------------ pool
struct PageRec {
  int32_t slot;
  int8_t tier;   // mkv_tier
};

struct SeqRec {
  int32_t len = 0;
  std::vector<PageRec> pages;
};

struct Staging {          // pinned host buffer + event guarding reuse
  void* host = nullptr;
  size_t bytes = 0;
  cudaEvent_t ev = nullptr;
  bool pending = false;
};

}  // namespace

struct mkv_pool {
  mkv_pool_config cfg{};
  bool host_only = false;
  int device = 0;
  int n_sm = 152;
  int G = 0;
  int64_t fp8_page_bytes = 0, tq3_page_bytes = 0;
  // device carve
  uint8_t* base = nullptr;
  size_t bytes = 0;
  uint8_t* fp8_arena = nullptr;
  uint8_t* tq3_arena = nullptr;
  uint8_t* plan_region = nullptr;
  size_t plan_bytes = 0;
  uint32_t* append_region = nullptr;
  int append_cap = 0;
  int2* demote_region = nullptr;
  int demote_cap = 0;
  float* workspace = nullptr;
  size_t workspace_bytes = 0;
  int* err = nullptr;
  int chunk_cap = 0;
  int entry_cap = 0;
  // host state
  std::vector<SeqRec> seqs;
  std::vector<int32_t> free_fp8, free_tq3;
  uint64_t generation = 1;
  uint64_t signs[4] = {0, 0, 0, 0};
  Lut lut{};
  // staging: two plan buffers, so that building a plan never waits for the
  // previous plan's upload (the device plan region is overwritten in stream
  // order, after the kernels that read it)
  Staging st_plan[2], st_append, st_demote;
  int plan_buf = 0;
  // plan cache
  uint64_t plan_gen = 0;
  std::vector<int32_t> plan_ids;
  int32_t plan_nq = 1;             // query tokens per request of the cached plan
  DecodeParams plan_params{};
  MergeParams merge_params{};
  int plan_parts = 0;
  int plan_entries = 0;             // page entries of the last plan built
  bool plan_injected = false;       // the device plan holds an injected entry (mkv_inject_plan_slot)
  std::vector<int32_t> plan_debug;   // kPlanRecord ints per chunk
  // one-shot timing events around the next decode kernel
  cudaEvent_t t_start = nullptr, t_stop = nullptr;
  // append cache (destinations in the append region)
  uint64_t app_gen = 0;
  std::vector<int32_t> app_ids, app_new;
  int app_ntok = 0;
  // fused append-decode destinations (same region)
};

namespace {

struct PlanLayout {
  size_t entries, groups, segs, merge, heads, total;
};

PlanLayout plan_layout(int entry_cap, int chunk_cap, int max_batch, int Hkv) {
  PlanLayout L;
  size_t off = 0;
  L.entries = off;
  off += align256(size_t(entry_cap) * sizeof(PageEntry));
  L.groups = off;
  off += align256(size_t(max_batch) * Hkv * 2 * sizeof(Group));
  L.segs = off;
  off += align256(size_t(chunk_cap) * sizeof(Segment));
  L.merge = off;
  off += align256(size_t(max_batch) * Hkv * sizeof(MergeDesc));
  L.heads = off;                         // per-CTA piece ranges (graph launches)
  off += align256(size_t(kMaxCtas + 1) * sizeof(int32_t));
  L.total = off;
  return L;
}

constexpr int kAppendCap = 65536;   // tokens per append launch
constexpr int kDemoteCap = 16384;   // pages per demote launch

int effective_batch(const mkv_pool_config& c) { return c.max_batch > 0 ? c.max_batch : c.max_seqs; }

mkv_status validate_config(const mkv_pool_config* c) {
  if (!c) return fail(MKV_ERR_INVALID_ARGUMENT, "config is NULL");
  if (c->num_layers < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1 || c->head_dim < 1 || c->page_size < 1 ||
      c->fp8_slots < 1 || c->tq3_slots < 0 || c->max_seqs < 1 || c->max_pages_per_seq < 1 || c->max_batch < 0)
    return fail(MKV_ERR_INVALID_ARGUMENT, "config fields must be positive");
  if (c->reserved != 0 || (c->flags & ~MKV_POOL_HOST_ONLY))
    return fail(MKV_ERR_INVALID_ARGUMENT, "unknown config flags / reserved field not 0");
  if (c->num_q_heads % c->num_kv_heads)
    return fail(MKV_ERR_INVALID_ARGUMENT, "num_q_heads must be a multiple of num_kv_heads");
  const int G = c->num_q_heads / c->num_kv_heads;
  if (G > kMaxGroup) return fail(MKV_ERR_UNSUPPORTED, "GQA group %d > %d", G, kMaxGroup);
  if (c->head_dim != kHeadDim) return fail(MKV_ERR_UNSUPPORTED, "head_dim %d: the kernels support 256", c->head_dim);
  if (c->page_size != 64 && c->page_size != 128)
    return fail(MKV_ERR_UNSUPPORTED, "page_size %d: supported 64 and 128", c->page_size);
  if (effective_batch(*c) > c->max_seqs) return fail(MKV_ERR_INVALID_ARGUMENT, "max_batch > max_seqs");
  if (int64_t(c->fp8_slots) >= (1 << 24) || int64_t(c->tq3_slots) >= (1 << 24))
    return fail(MKV_ERR_UNSUPPORTED, "slot counts must be < 2^24");
  return MKV_OK;
}

struct Sizes {
  int64_t fp8_page, tq3_page;
  size_t fp8_arena, tq3_arena, plan, append, demote, workspace, err, total;
  int entry_cap, chunk_cap;
};

Sizes compute_sizes(const mkv_pool_config& c) {
  Sizes s;
  const int P = c.page_size, H = c.num_kv_heads, D = c.head_dim;
  s.fp8_page = int64_t(H) * 2 * P * (D + 2);
  s.tq3_page = int64_t(H) * 2 * P * (3 * D / 8 + 2);
  s.fp8_arena = align256(size_t(c.num_layers) * c.fp8_slots * s.fp8_page);
  s.tq3_arena = align256(size_t(c.num_layers) * c.tq3_slots * s.tq3_page);
  const int mb = effective_batch(c);
  s.entry_cap = mb * c.max_pages_per_seq;
  s.chunk_cap = mb * H * 2 + 4 * kMaxCtas;
  s.plan = plan_layout(s.entry_cap, s.chunk_cap, mb, H).total;
  s.append = align256(size_t(kAppendCap) * 4);
  s.demote = align256(size_t(kDemoteCap) * 8);
  const int G = c.num_q_heads / c.num_kv_heads;
  // partial states: one per plan piece (at most chunk_cap), two per piece of
  // a paired multi-query plan
  s.workspace = align256(size_t(2) * s.chunk_cap * G * (2 + D) * 4);
  s.err = 256;
  s.total = s.fp8_arena + s.tq3_arena + s.plan + s.append + s.demote + s.workspace + s.err;
  return s;
}

mkv_status staging_alloc(Staging& st, size_t bytes) {
  st.bytes = bytes;
  cudaError_t e = cudaHostAlloc(&st.host, bytes, cudaHostAllocDefault);
  if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc");
  e = cudaEventCreateWithFlags(&st.ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
  return MKV_OK;
}

void staging_free(Staging& st) {
  if (st.ev) {
    cudaEventSynchronize(st.ev);
    cudaEventDestroy(st.ev);
  }
  if (st.host) cudaFreeHost(st.host);
  st = Staging{};
}

// Make the pinned buffer safe to overwrite (its previous copy has finished).
mkv_status staging_acquire(Staging& st) {
  if (st.pending) {
    const cudaError_t e = cudaEventSynchronize(st.ev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    st.pending = false;
  }
  return MKV_OK;
}

mkv_status staging_upload(Staging& st, void* dev, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return MKV_OK;
  cudaError_t e = cudaMemcpyAsync(dev, st.host, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (upload)");
  e = cudaEventRecord(st.ev, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  st.pending = true;
  return MKV_OK;
}

bool valid_seq(const mkv_pool* p, int32_t s) { return s >= 0 && s < p->cfg.max_seqs; }

int npages_for(int len, int P) { return (len + P - 1) / P; }

// ------------------------------------------------------------------ planner
// Relative cost of one token of one kv head, per format, plus a fixed cost per
// block and per piece, in units of one TQ3 token.  Fitted to per-CTA times of
// the decode kernel (GB300, 12 warps): a 32-token TQ3 block ~0.31 us of CTA
// time, a 16-token FP8 block ~0.25 us, a piece ~4 us (its end-of-piece merge
// and the warps' drift before it; set to 630 after the blocks got cheaper, by
// a sweep of step times on four workloads).  The planner works in integers,
// 1/100 of these units, so that its split is exact: a block costs
//   (20 per TQ3 token or 29 per FP8 token + 160) / 20 units,
// a round of n <= 12 blocks its slowest block times 12 (0.4 + 0.6 n / 12) =
// (24 + 3 n) / 5, and a piece 630.
constexpr int64_t kCostTq3Token = 20;    // 1.0 x 20
constexpr int64_t kCostFp8Token = 29;    // 1.45 x 20
constexpr int64_t kCostBlock = 160;      // 8 x 20
constexpr int64_t kCostPiece = 63000;    // 630 x 100
constexpr int kMinBlocksPerCta = 24;     // two blocks per warp at least
constexpr int kPlanRecord = 9;           // ints per split in mkv_plan_decode's output

// Split the batch's pages into groups (request, kv head, format), lay the
// groups' blocks out in one sequence, and cut that sequence into one
// contiguous piece list per CTA so that the largest CTA's estimated cost is
// as small as the cut points allow.  Each (CTA, group) piece
// writes one partial state; a group's partial states are contiguous, which is
// what the merge kernel reads.
mkv_status build_plan(mkv_pool* p, int32_t n_req, const int32_t* ids, int32_t nq, bool upload, cudaStream_t stream) {
  const int P = p->cfg.page_size, H = p->cfg.num_kv_heads;
  const PlanLayout L = plan_layout(p->entry_cap, p->chunk_cap, effective_batch(p->cfg), H);
  // One query token per request (nq = 1): entry b is request ids[b].  Several
  // (nq >= 2): the query tokens go in pairs, qpe = 2 per batch entry, which
  // the decode kernel serves from one dequantisation of each block; entry
  // b * npair + j (npair = ceil(nq / 2)) is request ids[b] cut after its query
  // token i1 = min(2j + 1, nq - 1), i.e. after its token len - nq + i1; query
  // token 2j sees that prefix but its last token (when 2j + 1 < nq).
  const int qpe = nq == 1 ? 1 : 2;
  const int npair = (nq + qpe - 1) / qpe;
  const int W = dec_warps(qpe);
  const int n = n_req * npair;
  if (n > effective_batch(p->cfg)) return fail(MKV_ERR_CAPACITY, "%d requests x %d query tokens > max_batch", n_req, nq);
  // planner costs: a paired block runs both query tokens' MMAs and softmax on
  // one dequantisation, and a paired piece ends with two merges
  const int64_t cost_tq3 = qpe == 1 ? kCostTq3Token : kCostTq3Token * 3 / 2;
  const int64_t cost_fp8 = qpe == 1 ? kCostFp8Token : kCostFp8Token * 3 / 2;
  const int64_t cost_piece = qpe == 1 ? kCostPiece : kCostPiece * 3 / 2;
  const int64_t round_full = 24 + 3 * int64_t(W);   // a round of W blocks, in units of its slowest block
  std::vector<PageEntry> entries;
  entries.reserve(size_t(n) * 64);
  struct BatchPages {
    int f_first, f_count, t_first, t_count;
  };
  std::vector<BatchPages> bp(n);
  for (int b = 0; b < n; ++b) {
    const SeqRec& s = p->seqs[ids[b / npair]];
    const int i1 = std::min(2 * (b % npair) + 1, nq - 1);
    const int len = s.len - (nq - 1 - i1);
    const int16_t tail = nq == 1 ? 1 : (2 * (b % npair) + 1 < nq ? kTailPairLast : 0);
    const int np = npages_for(len, P);
    BatchPages& B = bp[b];
    B.f_first = int(entries.size());
    for (int i = 0; i < np; ++i) {
      const int nv = (i == np - 1) ? len - i * P : P;
      if (s.pages[i].tier != MKV_TIER_STALE)
        entries.push_back({s.pages[i].slot, int16_t(nv), int16_t(i == np - 1 ? tail : 0)});
    }
    B.f_count = int(entries.size()) - B.f_first;
    B.t_first = int(entries.size());
    for (int i = 0; i < np; ++i)
      if (s.pages[i].tier == MKV_TIER_STALE) entries.push_back({s.pages[i].slot, int16_t(P), int16_t(0)});
    B.t_count = int(entries.size()) - B.t_first;
  }
  if (int(entries.size()) > p->entry_cap) return fail(MKV_ERR_CAPACITY, "plan entries exceed capacity");
  // groups, TQ3 before FP8 within each (request, kv head)
  std::vector<Group> groups;
  for (int b = 0; b < n; ++b)
    for (int kvh = 0; kvh < H; ++kvh)
      for (int fmt = 1; fmt >= 0; --fmt) {
        const int first = fmt ? bp[b].t_first : bp[b].f_first;
        const int count = fmt ? bp[b].t_count : bp[b].f_count;
        if (count == 0) continue;
        Group g{};
        g.b = b;
        g.kvh = kvh;
        g.fmt = fmt;
        g.entry0 = first;
        g.nentry = count;
        for (int i = 0; i < count; ++i) g.tokens += entries[first + i].nvalid;
        groups.push_back(g);
      }
  // Blocks: an FP8 block is kFp8Blk tokens and a TQ3 block kTq3Blk tokens
  // of one page; a group's blocks are numbered page by page, bpp = P / bt per
  // page, up to the last valid token (a block past a page's valid tokens is
  // empty and only costs its overhead).  Only a group's last page can be
  // partial, so a block's tokens never increase along the group.
  // Rounds: a CTA's W warps take a piece's blocks round-robin (block k of the
  // piece on warp k mod W), so a piece runs in rounds of up to W blocks from
  // its own first block on, and the next piece starts
  // after all of them.  A round costs its slowest block -- its first, since a
  // block's tokens never increase along a group -- on every warp; a short
  // round, with warps idle, runs its blocks faster and is priced between the
  // two.  Cuts may fall on any block.  A group's blocks are all alike but for
  // the last page's, so each group keeps the count and cost of its leading
  // full blocks.
  const int ng = int(groups.size());
  std::vector<int> g_nblk(ng), g_uni(ng);
  std::vector<int64_t> g_w(ng);
  auto blk_tokens = [&](const Group& g, int k) {
    const int bt = g.fmt ? kTq3Blk : kFp8Blk, bpp = P / bt;
    const int full = (g.nentry - 1) * bpp;
    if (k < full) return bt;
    return std::max(0, std::min(bt, int(entries[g.entry0 + g.nentry - 1].nvalid) - (k - full) * bt));
  };
  auto blk_cost = [&](int gi, int k) {
    const Group& g = groups[gi];
    return int64_t(blk_tokens(g, k)) * (g.fmt ? cost_tq3 : cost_fp8) + kCostBlock;
  };
  int64_t total_blocks = 0, lo = 0, hi = 0;
  for (int gi = 0; gi < ng; ++gi) {
    const Group& g = groups[gi];
    const int bt = g.fmt ? kTq3Blk : kFp8Blk;
    const int last_nv = entries[g.entry0 + g.nentry - 1].nvalid;
    g_nblk[gi] = (g.nentry - 1) * (P / bt) + (last_nv + bt - 1) / bt;
    g_uni[gi] = (g.nentry - 1) * (P / bt) + last_nv / bt;
    g_w[gi] = int64_t(bt) * (g.fmt ? cost_tq3 : cost_fp8) + kCostBlock;
    total_blocks += g_nblk[gi];
    // a CTA holds one block at least; the whole batch as one CTA fits hi
    lo = std::max(lo, cost_piece + blk_cost(gi, 0) * 27);
    hi += cost_piece + blk_cost(gi, 0) * round_full * ((g_nblk[gi] + W - 1) / W);
  }
  // The largest b1 in [b0, nblk] such that the piece [b0, b1) of group gi
  // costs at most `budget` (b0 when not one block fits); *cost gets its cost.
  // Whole rounds of full blocks are taken in O(1).
  auto piece_end = [&](int gi, int b0, int64_t budget, int64_t* cost) {
    const int nblk = g_nblk[gi], uni = g_uni[gi];
    int b = b0;
    int64_t used = 0;
    auto short_round = [&](int64_t worst, int avail) {   // blocks of a short round that fit what is left
      const int64_t left = budget - used;
      const int n = left >= 27 * worst ? int(std::min<int64_t>(avail - 1, (left / worst - 24) / 3)) : 0;
      b += n;
      used += n > 0 ? worst * (24 + 3 * int64_t(n)) : 0;
    };
    if (b < uni) {
      const int64_t w = g_w[gi], whole = (uni - b) / W;
      const int64_t take = std::min<int64_t>(whole, budget / (round_full * w));
      b += int(take) * W;
      used += take * round_full * w;
      if (take < whole) {       // the budget ends among full blocks
        short_round(w, W);
        *cost = used;
        return b;
      }
    }
    while (b < nblk) {
      const int64_t worst = blk_cost(gi, b);
      const int avail = std::min(W, nblk - b);
      if (used + worst * (24 + 3 * avail) > budget) {
        short_round(worst, avail);
        break;
      }
      used += worst * (24 + 3 * avail);
      b += avail;
    }
    *cost = used;
    return b;
  };
  // one CTA per SM at most, each with at least kMinBlocksPerCta blocks
  const int max_cta = int(std::max<int64_t>(
      1, std::min<int64_t>({int64_t(p->n_sm), int64_t(kMaxCtas), total_blocks / kMinBlocksPerCta})));
  // Contiguous split of the block sequence into at most max_cta CTAs that
  // minimises the largest CTA cost, a piece costing kCostPiece on top of its
  // rounds (its end-of-piece merge): the greedy fill below, which gives each
  // CTA the longest run that fits, needs the fewest CTAs for a given bound
  // (a run's cost only grows when it is extended and only falls when its
  // start moves later), so a bisection on the (integer) bound finds the
  // smallest one that fits.
  struct Cut {
    int group, blk;
  };
  // (it stops counting past max_cta CTAs)
  auto fill = [&](int64_t bound, std::vector<Cut>* starts) {
    int n_cta = 0;
    int64_t acc = 0;
    for (int gi = 0; gi < ng; ++gi)
      for (int b = 0; b < g_nblk[gi];) {
        int64_t c = 0;
        int b1 = (n_cta > 0 && acc + cost_piece < bound) ? piece_end(gi, b, bound - acc - cost_piece, &c) : b;
        if (b1 == b) {           // a new CTA takes the next block
          if (++n_cta > max_cta) return n_cta;
          if (starts) starts->push_back({gi, b});
          acc = 0;
          b1 = piece_end(gi, b, bound - cost_piece, &c);
          if (b1 == b) {         // below the one-block bound (not reached: bound >= lo)
            b1 = b + 1;
            c = blk_cost(gi, b) * 27;
          }
        }
        acc += cost_piece + c;
        b = b1;
      }
    return n_cta;
  };
  if (ng > 0 && fill(lo, nullptr) > max_cta) {
    // the smallest feasible bound: fill(hi) fits, fill(lo) does not
    while (hi - lo > 1) {
      const int64_t mid = lo + (hi - lo) / 2;
      (fill(mid, nullptr) <= max_cta ? hi : lo) = mid;
    }
    lo = hi;
  }
  std::vector<Cut> starts;
  const int ncta = ng == 0 ? 0 : fill(lo, &starts);
  starts.push_back({ng, 0});
  auto tokens_in = [&](const Group& g, int b0, int b1) {   // valid tokens of blocks [b0, b1)
    int64_t t = 0;
    const int bt = g.fmt ? kTq3Blk : kFp8Blk, full = (g.nentry - 1) * (P / bt);
    if (b0 < full) t += int64_t(std::min(b1, full) - b0) * bt;
    for (int k = std::max(b0, full); k < b1; ++k) t += blk_tokens(g, k);
    return int32_t(t);
  };
  std::vector<Segment> segs;
  std::vector<int32_t> seg_entry, seg_tokens;   // first page entry and valid tokens of each piece
  std::vector<int32_t> cta_seg(ncta + 1, 0);
  for (int c = 0; c < ncta; ++c) {
    cta_seg[c] = int(segs.size());
    const Cut from = starts[c], to = starts[c + 1];
    for (int gi = from.group; gi <= std::min(to.group, ng - 1); ++gi) {
      const int b0 = gi == from.group ? from.blk : 0;
      const int b1 = gi == to.group ? to.blk : g_nblk[gi];
      if (b1 <= b0) continue;
      const Group& g = groups[gi];
      Segment sg{};
      sg.fmt = g.fmt;
      sg.b = g.b;
      sg.kvh = g.kvh;
      sg.entry0 = g.entry0;
      sg.group = gi;
      sg.blk = b0;
      sg.nblk = b1 - b0;
      segs.push_back(sg);
      seg_entry.push_back(g.entry0 + b0 / (P / (g.fmt ? kTq3Blk : kFp8Blk)));
      seg_tokens.push_back(tokens_in(g, b0, b1));
    }
  }
  cta_seg[ncta] = int(segs.size());
  // (the workspace holds 2 chunk_cap partial states of G heads: qpe per piece)
  if (int(segs.size()) > p->chunk_cap) return fail(MKV_ERR_CAPACITY, "plan pieces exceed capacity");
  // partial-state indices: pieces are in group order, so each group's are contiguous
  for (Group& g : groups) g.nparts = 0;
  for (int i = 0; i < int(segs.size()); ++i) {
    Group& g = groups[segs[i].group];
    if (g.nparts == 0) g.part0 = i;
    segs[i].part = i;
    ++g.nparts;
  }
  std::vector<MergeDesc> md(size_t(n) * H, MergeDesc{0, 0, 0, 0});
  for (const Group& g : groups) {
    MergeDesc& m = md[size_t(g.b) * H + g.kvh];
    if (g.fmt) {
      m.tq3_first = g.part0;
      m.tq3_count = g.nparts;
    } else {
      m.fp8_first = g.part0;
      m.fp8_count = g.nparts;
    }
  }
  // debug record: one line per partial state (kPlanRecord ints)
  p->plan_debug.clear();
  for (int c = 0; c < ncta; ++c)
    for (int i = cta_seg[c]; i < cta_seg[c + 1]; ++i) {
      const Segment& sg = segs[i];
      const Group& g = groups[sg.group];
      const int bpp = P / (g.fmt ? kTq3Blk : kFp8Blk);
      const int last = g.entry0 + (sg.blk + sg.nblk - 1) / bpp;
      const int32_t rec[kPlanRecord] = {g.b, g.kvh, g.fmt ? 3 : 1, seg_entry[i], last - seg_entry[i] + 1,
                                        seg_tokens[i], c, sg.blk, sg.nblk};
      p->plan_debug.insert(p->plan_debug.end(), rec, rec + kPlanRecord);
    }
  p->plan_parts = int(segs.size());
  p->plan_entries = int(entries.size());
  p->plan_injected = false;
  // params
  DecodeParams& dp = p->plan_params;
  dp = DecodeParams{};
  dp.entries = reinterpret_cast<const PageEntry*>(p->plan_region + L.entries);
  dp.groups = reinterpret_cast<const Group*>(p->plan_region + L.groups);
  dp.segs = reinterpret_cast<const Segment*>(p->plan_region + L.segs);
  for (int i = 0; i <= ncta; ++i) dp.cta_seg[i] = cta_seg[i];
  for (int i = 0; i < ncta; ++i) dp.first[i] = cta_seg[i] < cta_seg[i + 1] ? segs[cta_seg[i]] : Segment{};
  dp.n_ctas = ncta;
  dp.fp8_page_bytes = p->fp8_page_bytes;
  dp.tq3_page_bytes = p->tq3_page_bytes;
  dp.fp8_slots = p->cfg.fp8_slots;
  dp.tq3_slots = p->cfg.tq3_slots;
  std::memcpy(dp.signs, p->signs, sizeof dp.signs);
  dp.Hq = p->cfg.num_q_heads;
  dp.Hkv = H;
  dp.G = p->G;
  dp.P = P;
  dp.part = p->workspace;
  dp.score_scale = float(1.4426950408889634 / std::sqrt(double(kHeadDim)));
  dp.lut = p->lut;
  dp.err = p->err;
  dp.qpe = qpe;
  dp.nq = nq;
  dp.npair = npair;
  MergeParams& mp = p->merge_params;
  mp = MergeParams{};
  mp.part = p->workspace;
  mp.desc = reinterpret_cast<const MergeDesc*>(p->plan_region + L.merge);
  mp.n = n;
  mp.Hq = p->cfg.num_q_heads;
  mp.Hkv = H;
  mp.G = p->G;
  mp.qpe = qpe;
  mp.nq = nq;
  mp.npair = npair;
  std::memcpy(mp.signs, p->signs, sizeof mp.signs);
  if (!upload) return MKV_OK;
  Staging& sp = p->st_plan[p->plan_buf];
  mkv_status st = staging_acquire(sp);
  if (st != MKV_OK) return st;
  p->plan_buf ^= 1;
  uint8_t* h = static_cast<uint8_t*>(sp.host);
  std::memcpy(h + L.entries, entries.data(), entries.size() * sizeof(PageEntry));
  std::memcpy(h + L.groups, groups.data(), groups.size() * sizeof(Group));
  std::memcpy(h + L.segs, segs.data(), segs.size() * sizeof(Segment));
  std::memcpy(h + L.merge, md.data(), md.size() * sizeof(MergeDesc));
  {
    int32_t* hd = reinterpret_cast<int32_t*>(h + L.heads);
    for (int i = 0; i <= kMaxCtas; ++i) hd[i] = cta_seg[std::min(i, ncta)];   // CTAs past ncta: no pieces
  }
  return staging_upload(sp, p->plan_region, L.total, stream);
}

// The decode plan of (ids, nq query tokens per request), rebuilt only when
// the pool changed or another batch was planned since.
mkv_status ensure_plan(mkv_pool* p, int32_t n, const int32_t* ids, int32_t nq, bool upload, cudaStream_t s) {
  const bool cached = p->plan_gen == p->generation && p->plan_nq == nq && p->plan_ids.size() == size_t(n) &&
                      std::equal(ids, ids + n, p->plan_ids.begin());
  if (cached) return MKV_OK;
  const mkv_status st = build_plan(p, n, ids, nq, upload, s);
  if (st != MKV_OK) {
    p->plan_gen = 0;
    return st;
  }
  p->plan_gen = p->generation;
  p->plan_nq = nq;
  p->plan_ids.assign(ids, ids + n);
  return MKV_OK;
}

// nq query tokens per request: each request holds at least nq tokens, the
// pages of its last nq tokens are FP8, and the plan's n * nq entries fit.
mkv_status check_queries(const mkv_pool* p, int32_t n, const int32_t* ids, int32_t nq) {
  if (nq < 1 || nq > effective_batch(p->cfg)) return fail(MKV_ERR_INVALID_ARGUMENT, "nq = %d", nq);
  if (int64_t(n) * nq > effective_batch(p->cfg))
    return fail(MKV_ERR_INVALID_ARGUMENT, "%d requests x %d query tokens > max_batch", n, nq);
  const int P = p->cfg.page_size;
  for (int i = 0; i < n; ++i) {
    const SeqRec& sr = p->seqs[ids[i]];
    if (sr.len < nq) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence %d holds %d < nq tokens", ids[i], sr.len);
    for (int pg = (sr.len - nq) / P; pg <= (sr.len - 1) / P; ++pg)
      if (sr.pages[pg].tier == MKV_TIER_STALE)
        return fail(MKV_ERR_INVALID_STATE, "sequence %d: a query token's page %d is TQ3", ids[i], pg);
  }
  return MKV_OK;
}

mkv_status check_batch(const mkv_pool* p, int32_t n, const int32_t* ids, bool need_nonempty) {
  if (n < 0 || (n > 0 && !ids)) return fail(MKV_ERR_INVALID_ARGUMENT, "bad batch");
  if (n > effective_batch(p->cfg)) return fail(MKV_ERR_INVALID_ARGUMENT, "batch %d > max_batch", n);
  std::vector<int32_t> sorted(ids, ids + n);
  std::sort(sorted.begin(), sorted.end());
  for (int i = 0; i < n; ++i) {
    if (!valid_seq(p, sorted[i])) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", sorted[i]);
    if (i && sorted[i] == sorted[i - 1]) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d repeated", sorted[i]);
    if (need_nonempty && p->seqs[sorted[i]].len == 0)
      return fail(MKV_ERR_INVALID_ARGUMENT, "sequence %d is empty", sorted[i]);
  }
  return MKV_OK;
}

}  // namespace

// ===================================================================== C ABI
extern "C" {

const char* mkv_last_error(void) { return g_last_error.c_str(); }

const char* mkv_version(void) { return "mkv 0.1.0 (sm_103a)"; }

mkv_status mkv_pool_required_bytes(const mkv_pool_config* cfg, size_t* device_bytes) {
  mkv_status st = validate_config(cfg);
  if (st != MKV_OK) return st;
  if (!device_bytes) return fail(MKV_ERR_INVALID_ARGUMENT, "device_bytes is NULL");
  *device_bytes = compute_sizes(*cfg).total;
  return MKV_OK;
}

mkv_status mkv_pool_create(const mkv_pool_config* cfg, void* device_buf, size_t bytes, mkv_stream_t stream,
                           mkv_pool** out) {
  mkv_status st = validate_config(cfg);
  if (st != MKV_OK) return st;
  if (!out) return fail(MKV_ERR_INVALID_ARGUMENT, "out is NULL");
  const bool host_only = (cfg->flags & MKV_POOL_HOST_ONLY) != 0;
  const Sizes S = compute_sizes(*cfg);
  if (!host_only) {
    if (!device_buf) return fail(MKV_ERR_INVALID_ARGUMENT, "device_buf is NULL");
    if (reinterpret_cast<uintptr_t>(device_buf) & 255) return fail(MKV_ERR_INVALID_ARGUMENT, "device_buf not 256-byte aligned");
    if (bytes < S.total) return fail(MKV_ERR_INVALID_ARGUMENT, "device buffer %zu < required %zu", bytes, S.total);
  }
  mkv_pool* p = new (std::nothrow) mkv_pool();
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "out of host memory");
  p->cfg = *cfg;
  p->host_only = host_only;
  p->G = cfg->num_q_heads / cfg->num_kv_heads;
  p->fp8_page_bytes = S.fp8_page;
  p->tq3_page_bytes = S.tq3_page;
  p->entry_cap = S.entry_cap;
  p->chunk_cap = S.chunk_cap;
  p->append_cap = kAppendCap;
  p->demote_cap = kDemoteCap;
  p->workspace_bytes = S.workspace;
  p->seqs.resize(cfg->max_seqs);
  for (int s = cfg->fp8_slots - 1; s >= 0; --s) p->free_fp8.push_back(s);
  for (int s = cfg->tq3_slots - 1; s >= 0; --s) p->free_tq3.push_back(s);
  uint64_t state = cfg->rotation_seed;
  for (int w = 0; w < 4; ++w) p->signs[w] = splitmix64_next(state);
  p->lut = make_lut(codebook());
  if (!host_only) {
    uint8_t* b = static_cast<uint8_t*>(device_buf);
    p->base = b;
    p->bytes = bytes;
    size_t off = 0;
    p->fp8_arena = b + off;
    off += S.fp8_arena;
    p->tq3_arena = b + off;
    off += S.tq3_arena;
    p->plan_region = b + off;
    p->plan_bytes = S.plan;
    off += S.plan;
    p->append_region = reinterpret_cast<uint32_t*>(b + off);
    off += S.append;
    p->demote_region = reinterpret_cast<int2*>(b + off);
    off += S.demote;
    p->workspace = reinterpret_cast<float*>(b + off);
    off += S.workspace;
    p->err = reinterpret_cast<int*>(b + off);
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->n_sm, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) {
      delete p;
      return cuda_fail(e, "device query");
    }
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(p->fp8_arena, 0, S.fp8_arena, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->err, 0, S.err, s);
    if (e != cudaSuccess) {
      delete p;
      return cuda_fail(e, "cudaMemsetAsync");
    }
    if ((st = staging_alloc(p->st_plan[0], S.plan)) != MKV_OK || (st = staging_alloc(p->st_plan[1], S.plan)) != MKV_OK ||
        (st = staging_alloc(p->st_append, S.append)) != MKV_OK || (st = staging_alloc(p->st_demote, S.demote)) != MKV_OK) {
      staging_free(p->st_plan[0]);
      staging_free(p->st_plan[1]);
      staging_free(p->st_append);
      staging_free(p->st_demote);
      delete p;
      return st;
    }
  }
  *out = p;
  return MKV_OK;
}

mkv_status mkv_pool_destroy(mkv_pool* p) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (!p->host_only) {
    staging_free(p->st_plan[0]);
    staging_free(p->st_plan[1]);
    staging_free(p->st_append);
    staging_free(p->st_demote);
  }
  delete p;
  return MKV_OK;
}

mkv_status mkv_seq_extend(mkv_pool* p, int32_t n, const int32_t* ids, const int32_t* n_new) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (n < 0 || (n > 0 && (!ids || !n_new))) return fail(MKV_ERR_INVALID_ARGUMENT, "bad arguments");
  const int P = p->cfg.page_size;
  std::vector<int32_t> seen(ids, ids + n);
  std::sort(seen.begin(), seen.end());
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    if (!valid_seq(p, ids[i])) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", ids[i]);
    if (i && seen[i] == seen[i - 1]) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d repeated", seen[i]);
    if (n_new[i] < 0) return fail(MKV_ERR_INVALID_ARGUMENT, "negative n_new");
    const SeqRec& s = p->seqs[ids[i]];
    const int64_t nl = int64_t(s.len) + n_new[i];
    if (nl > int64_t(p->cfg.max_pages_per_seq) * P)
      return fail(MKV_ERR_INVALID_ARGUMENT, "sequence %d would exceed max_pages_per_seq", ids[i]);
    need += npages_for(int(nl), P) - int64_t(s.pages.size());
  }
  if (need > int64_t(p->free_fp8.size()))
    return fail(MKV_ERR_OUT_OF_PAGES, "FP8 arena: need %lld free slots, have %zu", (long long)need, p->free_fp8.size());
  for (int i = 0; i < n; ++i) {
    SeqRec& s = p->seqs[ids[i]];
    s.len += n_new[i];
    const int np = npages_for(s.len, P);
    while (int(s.pages.size()) < np) {
      const int32_t slot = p->free_fp8.back();
      p->free_fp8.pop_back();
      s.pages.push_back({slot, int8_t(MKV_TIER_RECENT)});
    }
  }
  if (n) ++p->generation;
  return MKV_OK;
}

mkv_status mkv_seq_release(mkv_pool* p, int32_t seq) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (!valid_seq(p, seq)) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", seq);
  SeqRec& s = p->seqs[seq];
  for (const PageRec& r : s.pages) (r.tier == MKV_TIER_STALE ? p->free_tq3 : p->free_fp8).push_back(r.slot);
  s.pages.clear();
  s.len = 0;
  ++p->generation;
  return MKV_OK;
}

mkv_status mkv_seq_info(const mkv_pool* p, int32_t seq, int32_t* length, int32_t* num_pages) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (!valid_seq(p, seq)) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", seq);
  if (length) *length = p->seqs[seq].len;
  if (num_pages) *num_pages = int32_t(p->seqs[seq].pages.size());
  return MKV_OK;
}

mkv_status mkv_page_info(const mkv_pool* p, int32_t seq, int32_t page, mkv_tier* tier, int32_t* slot) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (!valid_seq(p, seq)) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", seq);
  const SeqRec& s = p->seqs[seq];
  if (page < 0 || page >= int(s.pages.size())) return fail(MKV_ERR_INVALID_ARGUMENT, "page %d out of range", page);
  if (tier) *tier = mkv_tier(s.pages[page].tier);
  if (slot) *slot = s.pages[page].slot;
  return MKV_OK;
}

mkv_status mkv_append_tokens(mkv_pool* p, int32_t layer, int32_t n, const int32_t* ids, const int32_t* n_new,
                             const void* k, const void* v, mkv_dtype dtype, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if (dtype != MKV_F32 && dtype != MKV_BF16) return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  mkv_status st = check_batch(p, n, ids, false);
  if (st != MKV_OK) return st;
  if (n > 0 && !n_new) return fail(MKV_ERR_INVALID_ARGUMENT, "n_new is NULL");
  const int P = p->cfg.page_size;
  int64_t ntok = 0;
  for (int i = 0; i < n; ++i) {
    const SeqRec& s = p->seqs[ids[i]];
    if (n_new[i] < 0 || n_new[i] > s.len)
      return fail(MKV_ERR_INVALID_ARGUMENT, "n_new[%d] = %d outside [0, length %d]", i, n_new[i], s.len);
    for (int pos = s.len - n_new[i]; pos < s.len; pos += P - (pos % P)) {
      if (s.pages[pos / P].tier == MKV_TIER_STALE)
        return fail(MKV_ERR_INVALID_STATE, "sequence %d page %d is TQ3; append writes FP8 pages", ids[i], pos / P);
    }
    ntok += n_new[i];
  }
  if (ntok > 0 && (!k || !v)) return fail(MKV_ERR_INVALID_ARGUMENT, "k or v is NULL");
  if (ntok == 0 || p->host_only) return MKV_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // destinations (cached across layers for the same batch and pool state)
  const bool cached = p->app_gen == p->generation && p->app_ntok == ntok && p->app_ids.size() == size_t(n) &&
                      std::equal(ids, ids + n, p->app_ids.begin()) && std::equal(n_new, n_new + n, p->app_new.begin());
  std::vector<uint32_t> dest;
  if (!cached || ntok > p->append_cap) {
    dest.reserve(size_t(ntok));
    for (int i = 0; i < n; ++i) {
      const SeqRec& sq = p->seqs[ids[i]];
      for (int pos = sq.len - n_new[i]; pos < sq.len; ++pos)
        dest.push_back((uint32_t(sq.pages[pos / P].slot) << 8) | uint32_t(pos % P));
    }
  }
  AppendParams ap{};
  ap.fp8_layer = p->fp8_arena + int64_t(layer) * p->cfg.fp8_slots * p->fp8_page_bytes;
  ap.fp8_page_bytes = p->fp8_page_bytes;
  ap.kv_bf16 = dtype == MKV_BF16;
  ap.Hkv = p->cfg.num_kv_heads;
  ap.P = P;
  const size_t elt = dtype == MKV_BF16 ? 2 : 4;
  const size_t row = size_t(p->cfg.num_kv_heads) * kHeadDim * elt;
  for (int64_t t0 = 0; t0 < ntok; t0 += p->append_cap) {
    const int cnt = int(std::min<int64_t>(p->append_cap, ntok - t0));
    if (!(cached && ntok <= p->append_cap)) {
      if ((st = staging_acquire(p->st_append)) != MKV_OK) return st;
      std::memcpy(p->st_append.host, dest.data() + t0, size_t(cnt) * 4);
      if ((st = staging_upload(p->st_append, p->append_region, size_t(cnt) * 4, s)) != MKV_OK) return st;
    }
    ap.dest = p->append_region;
    ap.k = static_cast<const uint8_t*>(k) + t0 * row;
    ap.v = static_cast<const uint8_t*>(v) + t0 * row;
    ap.ntok = cnt;
    const cudaError_t e = launch_append(ap, s);
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
  }
  if (ntok <= p->append_cap) {
    p->app_gen = p->generation;
    p->app_ntok = int(ntok);
    p->app_ids.assign(ids, ids + n);
    p->app_new.assign(n_new, n_new + n);
  } else {
    p->app_gen = 0;
  }
  return MKV_OK;
}

mkv_status mkv_set_tier(mkv_pool* p, int32_t seq, int32_t page, mkv_tier tier) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (!valid_seq(p, seq)) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", seq);
  SeqRec& s = p->seqs[seq];
  if (page < 0 || page >= int(s.pages.size())) return fail(MKV_ERR_INVALID_ARGUMENT, "page %d out of range", page);
  if (tier != MKV_TIER_RECENT && tier != MKV_TIER_ANCHOR && tier != MKV_TIER_STALE)
    return fail(MKV_ERR_INVALID_ARGUMENT, "tier %d", int(tier));
  if (tier == MKV_TIER_STALE) return fail(MKV_ERR_INVALID_STATE, "use mkv_demote_pages to make a page STALE");
  if (s.pages[page].tier == MKV_TIER_STALE)
    return fail(MKV_ERR_INVALID_STATE, "page %d of sequence %d is TQ3; only FP8 pages change tier", page, seq);
  s.pages[page].tier = int8_t(tier);
  return MKV_OK;
}

mkv_status mkv_demote_pages(mkv_pool* p, int32_t n, const int32_t* ids, const int32_t* pages, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (n < 0 || (n > 0 && (!ids || !pages))) return fail(MKV_ERR_INVALID_ARGUMENT, "bad arguments");
  const int P = p->cfg.page_size;
  std::vector<std::pair<int32_t, int32_t>> seen;
  for (int i = 0; i < n; ++i) {
    if (!valid_seq(p, ids[i])) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", ids[i]);
    const SeqRec& s = p->seqs[ids[i]];
    if (pages[i] < 0 || pages[i] >= int(s.pages.size()))
      return fail(MKV_ERR_INVALID_ARGUMENT, "page %d of sequence %d out of range", pages[i], ids[i]);
    const PageRec& r = s.pages[pages[i]];
    if (r.tier == MKV_TIER_ANCHOR)
      return fail(MKV_ERR_INVALID_STATE, "page %d of sequence %d is an Anchor", pages[i], ids[i]);
    if (r.tier == MKV_TIER_STALE)
      return fail(MKV_ERR_INVALID_STATE, "page %d of sequence %d is already TQ3", pages[i], ids[i]);
    if (int64_t(pages[i] + 1) * P > s.len)
      return fail(MKV_ERR_INVALID_STATE, "page %d of sequence %d is not full", pages[i], ids[i]);
    seen.push_back({ids[i], pages[i]});
  }
  std::sort(seen.begin(), seen.end());
  for (size_t i = 1; i < seen.size(); ++i)
    if (seen[i] == seen[i - 1]) return fail(MKV_ERR_INVALID_STATE, "page listed twice");
  if (int64_t(n) > int64_t(p->free_tq3.size()))
    return fail(MKV_ERR_OUT_OF_PAGES, "TQ3 arena: need %d free slots, have %zu", n, p->free_tq3.size());
  if (n == 0) return MKV_OK;
  std::vector<int2> pairs(n);
  for (int i = 0; i < n; ++i) {
    pairs[i].x = p->seqs[ids[i]].pages[pages[i]].slot;
    pairs[i].y = p->free_tq3[p->free_tq3.size() - 1 - i];
  }
  if (!p->host_only) {
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DemoteParams dp{};
    dp.fp8_arena = p->fp8_arena;
    dp.tq3_arena = p->tq3_arena;
    dp.fp8_page_bytes = p->fp8_page_bytes;
    dp.tq3_page_bytes = p->tq3_page_bytes;
    dp.fp8_layer_stride = int64_t(p->cfg.fp8_slots) * p->fp8_page_bytes;
    dp.tq3_layer_stride = int64_t(p->cfg.tq3_slots) * p->tq3_page_bytes;
    dp.L = p->cfg.num_layers;
    dp.Hkv = p->cfg.num_kv_heads;
    dp.P = P;
    std::memcpy(dp.signs, p->signs, sizeof dp.signs);
    std::memcpy(dp.thr, codebook().thr, sizeof dp.thr);
    for (int i0 = 0; i0 < n; i0 += p->demote_cap) {
      const int cnt = std::min(p->demote_cap, n - i0);
      mkv_status st = staging_acquire(p->st_demote);
      if (st != MKV_OK) return st;
      std::memcpy(p->st_demote.host, pairs.data() + i0, size_t(cnt) * sizeof(int2));
      if ((st = staging_upload(p->st_demote, p->demote_region, size_t(cnt) * sizeof(int2), s)) != MKV_OK) return st;
      dp.pairs = p->demote_region;
      dp.npairs = cnt;
      const cudaError_t e = launch_demote(dp, s);
      if (e != cudaSuccess) return cuda_fail(e, "demote launch");
    }
  }
  for (int i = 0; i < n; ++i) {
    PageRec& r = p->seqs[ids[i]].pages[pages[i]];
    p->free_fp8.push_back(r.slot);
    r.slot = pairs[i].y;
    r.tier = int8_t(MKV_TIER_STALE);
  }
  p->free_tq3.resize(p->free_tq3.size() - n);
  ++p->generation;
  return MKV_OK;
}

// Enqueue the decode kernel (with the fused append when k is non-NULL) and
// the merge for the pool's current plan; partial states go to `part`.
mkv_status enqueue_decode(mkv_pool* p, int32_t layer, const void* q, mkv_dtype q_dtype, float* part, const void* k,
                          const void* v, mkv_dtype kv_dtype, float* out, float* lse, cudaStream_t s,
                          bool fixed_params = false) {
  DecodeParams dp = p->plan_params;
  if (fixed_params) {
    // parameters that stay valid for every later plan: the CTAs read their
    // piece ranges from the plan region, and the grid is one CTA per SM
    const PlanLayout L = plan_layout(p->entry_cap, p->chunk_cap, effective_batch(p->cfg), p->cfg.num_kv_heads);
    dp.heads = reinterpret_cast<const int32_t*>(p->plan_region + L.heads);
    dp.n_ctas = std::min(p->n_sm, kMaxCtas);
  }
  dp.fp8_layer = p->fp8_arena + int64_t(layer) * p->cfg.fp8_slots * p->fp8_page_bytes;
  dp.tq3_layer = p->tq3_arena + int64_t(layer) * p->cfg.tq3_slots * p->tq3_page_bytes;
  dp.q = q;
  dp.q_bf16 = q_dtype == MKV_BF16;
  dp.part = part;
  dp.append = k != nullptr;
  dp.kv_bf16 = kv_dtype == MKV_BF16;
  dp.k = k;
  dp.v = v;
  cudaError_t e = cudaSuccess;
  if (p->t_start) e = cudaEventRecord(p->t_start, s);
  if (e == cudaSuccess) e = launch_decode(dp, s);
  if (e == cudaSuccess && p->t_stop) e = cudaEventRecord(p->t_stop, s);
  p->t_start = p->t_stop = nullptr;
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  MergeParams mp = p->merge_params;
  mp.part = part;
  mp.out = out;
  mp.lse = lse;
  e = launch_merge(mp, s);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return MKV_OK;
}

mkv_status mkv_decode_attention(mkv_pool* p, int32_t layer, int32_t n, const int32_t* ids, const void* q,
                                mkv_dtype dtype, float* out, float* lse, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if (dtype != MKV_F32 && dtype != MKV_BF16) return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  mkv_status st = check_batch(p, n, ids, true);
  if (st != MKV_OK) return st;
  if (n == 0) return MKV_OK;
  if (!q || !out || !lse) return fail(MKV_ERR_INVALID_ARGUMENT, "q/out/lse is NULL");
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = ensure_plan(p, n, ids, 1, !p->host_only, s)) != MKV_OK) return st;
  if (p->host_only) return MKV_OK;
  return enqueue_decode(p, layer, q, dtype, p->workspace, nullptr, nullptr, MKV_F32, out, lse, s);
}

mkv_status mkv_decode_attention_multi(mkv_pool* p, int32_t layer, int32_t n, const int32_t* ids, int32_t nq,
                                      const void* q, mkv_dtype dtype, float* out, float* lse, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if (dtype != MKV_F32 && dtype != MKV_BF16) return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  mkv_status st = check_batch(p, n, ids, true);
  if (st != MKV_OK) return st;
  if ((st = check_queries(p, n, ids, nq)) != MKV_OK) return st;
  if (n == 0) return MKV_OK;
  if (!q || !out || !lse) return fail(MKV_ERR_INVALID_ARGUMENT, "q/out/lse is NULL");
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = ensure_plan(p, n, ids, nq, !p->host_only, s)) != MKV_OK) return st;
  if (p->host_only) return MKV_OK;
  return enqueue_decode(p, layer, q, dtype, p->workspace, nullptr, nullptr, MKV_F32, out, lse, s);
}

// Same as mkv_decode_attention, with the partial states in the library's fixed
// device scratch instead of the pool workspace; allocates nothing.
mkv_status mkv_decode_attention_noalloc(mkv_pool* p, int32_t layer, int32_t n, const int32_t* ids, const void* q,
                                        mkv_dtype dtype, float* out, float* lse, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if (dtype != MKV_F32 && dtype != MKV_BF16) return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  mkv_status st = check_batch(p, n, ids, true);
  if (st != MKV_OK) return st;
  if (n == 0) return MKV_OK;
  if (!q || !out || !lse) return fail(MKV_ERR_INVALID_ARGUMENT, "q/out/lse is NULL");
  if (p->host_only) return fail(MKV_ERR_UNSUPPORTED, "host-only pool: no device scratch");
  // the scratch address is per device: it must be the pool's
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != p->device)
    return fail(MKV_ERR_INVALID_ARGUMENT, "current device %d is not the pool's device %d", cur, p->device);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = ensure_plan(p, n, ids, 1, true, s)) != MKV_OK) return st;
  float* scratch = nullptr;
  size_t scratch_bytes = 0;
  e = noalloc_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "device scratch address (cudaGetSymbolAddress)");
  // scratch = the partial states
  const size_t need = size_t(p->plan_parts) * p->G * (2 + kHeadDim) * sizeof(float);
  if (need > scratch_bytes)
    return fail(MKV_ERR_CAPACITY, "batch needs %zu bytes of scratch; the fixed scratch holds %zu", need,
                scratch_bytes);
  return enqueue_decode(p, layer, q, dtype, scratch, nullptr, nullptr, MKV_F32, out, lse, s);
}

mkv_status mkv_append_decode(mkv_pool* p, int32_t layer, int32_t n, const int32_t* ids, const void* k,
                             const void* v, mkv_dtype kv_dtype, const void* q, mkv_dtype q_dtype, float* out,
                             float* lse, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if ((kv_dtype != MKV_F32 && kv_dtype != MKV_BF16) || (q_dtype != MKV_F32 && q_dtype != MKV_BF16))
    return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  mkv_status st = check_batch(p, n, ids, true);
  if (st != MKV_OK) return st;
  if (n == 0) return MKV_OK;
  if (!k || !v || !q || !out || !lse) return fail(MKV_ERR_INVALID_ARGUMENT, "k/v/q/out/lse is NULL");
  const int P = p->cfg.page_size;
  for (int i = 0; i < n; ++i) {
    const SeqRec& s = p->seqs[ids[i]];
    if (s.pages[(s.len - 1) / P].tier == MKV_TIER_STALE)
      return fail(MKV_ERR_INVALID_STATE, "sequence %d: the newest token's page is TQ3", ids[i]);
  }
  if (p->host_only) return MKV_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->plan_injected) p->plan_gen = 0;   // the fused append writes through the plan's slots: replan
  if ((st = ensure_plan(p, n, ids, 1, true, s)) != MKV_OK) return st;
  return enqueue_decode(p, layer, q, q_dtype, p->workspace, k, v, kv_dtype, out, lse, s);
}

// ------------------------------------------------------------------ page relevance
mkv_status mkv_page_relevance(mkv_pool* p, int32_t layer, int32_t n, const int32_t* ids, const void* q,
                              mkv_dtype q_dtype, const float* lse, float* mass, int32_t mass_stride,
                              mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if (q_dtype != MKV_F32 && q_dtype != MKV_BF16) return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  mkv_status st = check_batch(p, n, ids, true);
  if (st != MKV_OK) return st;
  if (n == 0) return MKV_OK;
  if (!q || !lse || !mass) return fail(MKV_ERR_INVALID_ARGUMENT, "q/lse/mass is NULL");
  const int P = p->cfg.page_size;
  int max_pages = 0;
  for (int i = 0; i < n; ++i) max_pages = std::max(max_pages, npages_for(p->seqs[ids[i]].len, P));
  if (mass_stride < max_pages)
    return fail(MKV_ERR_INVALID_ARGUMENT, "mass_stride %d < %d pages of the longest sequence", mass_stride, max_pages);
  if (p->host_only) return MKV_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  RelevanceParams rp{};
  rp.fp8_layer = p->fp8_arena + int64_t(layer) * p->cfg.fp8_slots * p->fp8_page_bytes;
  rp.tq3_layer = p->tq3_arena + int64_t(layer) * p->cfg.tq3_slots * p->tq3_page_bytes;
  rp.fp8_page_bytes = p->fp8_page_bytes;
  rp.tq3_page_bytes = p->tq3_page_bytes;
  rp.pages = reinterpret_cast<const int4*>(p->demote_region);
  rp.Hq = p->cfg.num_q_heads;
  rp.Hkv = p->cfg.num_kv_heads;
  rp.G = p->G;
  rp.P = P;
  rp.q = q;
  rp.q_bf16 = q_dtype == MKV_BF16;
  rp.lse = lse;
  rp.mass = mass;
  rp.mass_stride = mass_stride;
  std::memcpy(rp.signs, p->signs, sizeof rp.signs);
  std::memcpy(rp.level, codebook().level, sizeof rp.level);
  // the (request, page) list goes through the demotion staging region, as
  // many int4 records per launch as its int2 capacity holds
  const int cap = p->demote_cap / 2;
  std::vector<int4> list;
  for (int i = 0; i < n; ++i) {
    const SeqRec& sr = p->seqs[ids[i]];
    const int np = npages_for(sr.len, P);
    for (int pg = 0; pg < np; ++pg)
      list.push_back(make_int4(i, pg, sr.pages[pg].slot, (int(sr.pages[pg].tier) << 16) | std::min(P, sr.len - pg * P)));
  }
  for (size_t at = 0; at < list.size(); at += cap) {
    const int cnt = int(std::min<size_t>(cap, list.size() - at));
    if ((st = staging_acquire(p->st_demote)) != MKV_OK) return st;
    std::memcpy(p->st_demote.host, list.data() + at, size_t(cnt) * sizeof(int4));
    if ((st = staging_upload(p->st_demote, p->demote_region, size_t(cnt) * sizeof(int4), s)) != MKV_OK) return st;
    rp.npages = cnt;
    const cudaError_t e = launch_relevance(rp, s);
    if (e != cudaSuccess) return cuda_fail(e, "relevance launch");
  }
  return MKV_OK;
}

// ------------------------------------------------------------------ step graph
struct mkv_step_graph {
  mkv_pool* pool = nullptr;
  std::vector<int32_t> ids;
  bool append = false;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

mkv_status mkv_step_graph_create(mkv_pool* p, int32_t n, const int32_t* ids, const void* const* q,
                                 const void* const* k, const void* const* v, mkv_dtype q_dtype, mkv_dtype kv_dtype,
                                 float* const* out, float* const* lse, mkv_stream_t stream, mkv_step_graph** graph) {
  if (!p || !graph) return fail(MKV_ERR_INVALID_ARGUMENT, "pool or graph is NULL");
  *graph = nullptr;
  if (p->host_only) return fail(MKV_ERR_UNSUPPORTED, "host-only pool: no graph");
  if ((q_dtype != MKV_F32 && q_dtype != MKV_BF16) || (kv_dtype != MKV_F32 && kv_dtype != MKV_BF16))
    return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  mkv_status st = check_batch(p, n, ids, true);
  if (st != MKV_OK) return st;
  if (n == 0) return fail(MKV_ERR_INVALID_ARGUMENT, "empty batch");
  const int L = p->cfg.num_layers;
  if (!q || !out || !lse || (!k) != (!v)) return fail(MKV_ERR_INVALID_ARGUMENT, "q/out/lse (or one of k, v) is NULL");
  for (int l = 0; l < L; ++l)
    if (!q[l] || !out[l] || !lse[l] || (k && (!k[l] || !v[l])))
      return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d: a buffer pointer is NULL", l);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (k) {
    const int P = p->cfg.page_size;
    for (int i = 0; i < n; ++i) {
      const SeqRec& sr = p->seqs[ids[i]];
      if (sr.pages[(sr.len - 1) / P].tier == MKV_TIER_STALE)
        return fail(MKV_ERR_INVALID_STATE, "sequence %d: the newest token's page is TQ3", ids[i]);
    }
  }
  if (p->plan_injected) p->plan_gen = 0;
  if ((st = ensure_plan(p, n, ids, 1, true, s)) != MKV_OK) return st;
  // the kernels' shared-memory limit is a per-device attribute, set outside the capture
  cudaError_t e = prepare_decode_launch();
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel attribute");
  auto* g = new mkv_step_graph;
  g->pool = p;
  g->ids.assign(ids, ids + n);
  g->append = k != nullptr;
  // record on a private stream (the caller's may be the legacy default
  // stream, which cannot be captured); the recording executes nothing
  cudaStream_t cap = nullptr;
  e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    delete g;
    return cuda_fail(e, "cudaStreamCreate");
  }
  e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cap);
    delete g;
    return cuda_fail(e, "cudaStreamBeginCapture");
  }
  void* t_start = p->t_start;
  void* t_stop = p->t_stop;
  p->t_start = p->t_stop = nullptr;     // timing events are not part of a graph
  mkv_status rec = MKV_OK;
  for (int l = 0; l < L && rec == MKV_OK; ++l)
    rec = enqueue_decode(p, l, q[l], q_dtype, p->workspace, k ? k[l] : nullptr, k ? v[l] : nullptr, kv_dtype, out[l],
                         lse[l], cap, true);
  p->t_start = static_cast<cudaEvent_t>(t_start);
  p->t_stop = static_cast<cudaEvent_t>(t_stop);
  e = cudaStreamEndCapture(cap, &g->graph);
  cudaStreamDestroy(cap);
  if (rec != MKV_OK || e != cudaSuccess) {
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    return rec != MKV_OK ? rec : cuda_fail(e, "cudaStreamEndCapture");
  }
  e = cudaGraphInstantiate(&g->exec, g->graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g->graph);
    delete g;
    return cuda_fail(e, "cudaGraphInstantiate");
  }
  *graph = g;
  return MKV_OK;
}

mkv_status mkv_step_graph_launch(mkv_step_graph* g, mkv_stream_t stream) {
  if (!g) return fail(MKV_ERR_INVALID_ARGUMENT, "graph is NULL");
  mkv_pool* p = g->pool;
  const int n = int(g->ids.size());
  mkv_status st = check_batch(p, n, g->ids.data(), true);
  if (st != MKV_OK) return st;
  if (g->append) {
    const int P = p->cfg.page_size;
    for (int i = 0; i < n; ++i) {
      const SeqRec& sr = p->seqs[g->ids[i]];
      if (sr.pages[(sr.len - 1) / P].tier == MKV_TIER_STALE)
        return fail(MKV_ERR_INVALID_STATE, "sequence %d: the newest token's page is TQ3", g->ids[i]);
    }
  }
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->plan_injected) p->plan_gen = 0;
  // the plan (re-)uploaded here in stream order is what the graph's kernels read
  if ((st = ensure_plan(p, n, g->ids.data(), 1, true, s)) != MKV_OK) return st;
  const cudaError_t e = cudaGraphLaunch(g->exec, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  return MKV_OK;
}

mkv_status mkv_step_graph_destroy(mkv_step_graph* g) {
  if (!g) return fail(MKV_ERR_INVALID_ARGUMENT, "graph is NULL");
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
  return MKV_OK;
}

mkv_status mkv_dequantize_pages(mkv_pool* p, int32_t layer, int32_t seq, int32_t page0, int32_t npages,
                                void* k_out, void* v_out, mkv_dtype out_dtype, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if (!valid_seq(p, seq)) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", seq);
  if (out_dtype != MKV_F32 && out_dtype != MKV_BF16) return fail(MKV_ERR_INVALID_ARGUMENT, "dtype");
  const SeqRec& s = p->seqs[seq];
  if (npages < 0 || page0 < 0 || page0 + npages > int(s.pages.size()))
    return fail(MKV_ERR_INVALID_ARGUMENT, "page range [%d, %d) outside the sequence's %zu pages", page0,
                page0 + npages, s.pages.size());
  if (npages == 0) return MKV_OK;
  if (!k_out || !v_out) return fail(MKV_ERR_INVALID_ARGUMENT, "k_out/v_out is NULL");
  if (npages > p->demote_cap) return fail(MKV_ERR_CAPACITY, "at most %d pages per call", p->demote_cap);
  if (p->host_only) return MKV_OK;
  const int P = p->cfg.page_size;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  mkv_status r = staging_acquire(p->st_demote);
  if (r != MKV_OK) return r;
  int2* h = static_cast<int2*>(p->st_demote.host);
  for (int i = 0; i < npages; ++i) {
    const PageRec& rec = s.pages[page0 + i];
    const int nv = std::min(P, s.len - (page0 + i) * P);
    h[i].x = rec.slot;
    h[i].y = (int(rec.tier) << 16) | nv;
  }
  if ((r = staging_upload(p->st_demote, p->demote_region, size_t(npages) * sizeof(int2), st)) != MKV_OK) return r;
  DequantParams dq{};
  dq.fp8_layer = p->fp8_arena + int64_t(layer) * p->cfg.fp8_slots * p->fp8_page_bytes;
  dq.tq3_layer = p->tq3_arena + int64_t(layer) * p->cfg.tq3_slots * p->tq3_page_bytes;
  dq.fp8_page_bytes = p->fp8_page_bytes;
  dq.tq3_page_bytes = p->tq3_page_bytes;
  dq.pages = p->demote_region;
  dq.npages = npages;
  dq.Hkv = p->cfg.num_kv_heads;
  dq.P = P;
  dq.out_bf16 = out_dtype == MKV_BF16;
  dq.k_out = k_out;
  dq.v_out = v_out;
  std::memcpy(dq.signs, p->signs, sizeof dq.signs);
  std::memcpy(dq.level, codebook().level, sizeof dq.level);
  const cudaError_t e = launch_dequant(dq, st);
  if (e != cudaSuccess) return cuda_fail(e, "dequantise launch");
  return MKV_OK;
}

mkv_status mkv_pool_stats(const mkv_pool* p, mkv_stats* out) {
  if (!p || !out) return fail(MKV_ERR_INVALID_ARGUMENT, "NULL argument");
  mkv_stats st{};
  for (const SeqRec& s : p->seqs) {
    st.live_tokens += s.len;
    for (const PageRec& r : s.pages) {
      if (r.tier == MKV_TIER_RECENT) ++st.recent_pages;
      if (r.tier == MKV_TIER_ANCHOR) ++st.anchor_pages;
      if (r.tier == MKV_TIER_STALE) ++st.stale_pages;
    }
  }
  const int64_t L = p->cfg.num_layers;
  st.fp8_bytes = (st.recent_pages + st.anchor_pages) * p->fp8_page_bytes * L;
  st.tq3_bytes = st.stale_pages * p->tq3_page_bytes * L;
  st.kv_bytes_per_live_token = st.live_tokens ? double(st.fp8_bytes + st.tq3_bytes) / double(st.live_tokens) : 0.0;
  st.fp8_slots_free = int32_t(p->free_fp8.size());
  st.tq3_slots_free = int32_t(p->free_tq3.size());
  st.device_bytes = int64_t(compute_sizes(p->cfg).total);
  st.workspace_bytes = int64_t(p->workspace_bytes);
  *out = st;
  return MKV_OK;
}

mkv_status mkv_export_page(mkv_pool* p, int32_t layer, int32_t seq, int32_t page, void* host_dst, size_t cap,
                           mkv_tier* tier, int32_t* n_valid, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (layer < 0 || layer >= p->cfg.num_layers) return fail(MKV_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  if (!valid_seq(p, seq)) return fail(MKV_ERR_INVALID_ARGUMENT, "sequence id %d out of range", seq);
  const SeqRec& s = p->seqs[seq];
  if (page < 0 || page >= int(s.pages.size())) return fail(MKV_ERR_INVALID_ARGUMENT, "page %d out of range", page);
  const PageRec r = s.pages[page];
  const bool tq3 = r.tier == MKV_TIER_STALE;
  const int64_t pb = tq3 ? p->tq3_page_bytes : p->fp8_page_bytes;
  if (tier) *tier = mkv_tier(r.tier);
  if (n_valid) *n_valid = std::min(p->cfg.page_size, s.len - page * p->cfg.page_size);
  if (!host_dst || cap < size_t(pb)) return fail(MKV_ERR_INVALID_ARGUMENT, "host_dst too small (%lld bytes needed)", (long long)pb);
  if (p->host_only) return fail(MKV_ERR_UNSUPPORTED, "host-only pool has no page bytes");
  const uint8_t* src = (tq3 ? p->tq3_arena + int64_t(layer) * p->cfg.tq3_slots * pb
                            : p->fp8_arena + int64_t(layer) * p->cfg.fp8_slots * pb) +
                       int64_t(r.slot) * pb;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_dst, src, size_t(pb), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "export copy");
  return MKV_OK;
}

mkv_status mkv_rotation_signs(const mkv_pool* p, int8_t* dst, int32_t cap) {
  if (!p || !dst) return fail(MKV_ERR_INVALID_ARGUMENT, "NULL argument");
  if (cap < p->cfg.head_dim) return fail(MKV_ERR_INVALID_ARGUMENT, "cap < head_dim");
  for (int i = 0; i < p->cfg.head_dim; ++i) dst[i] = ((p->signs[i >> 6] >> (i & 63)) & 1) ? -1 : 1;
  return MKV_OK;
}

mkv_status mkv_tq3_codebook(float* levels8, float* thresholds7) {
  if (!levels8 || !thresholds7) return fail(MKV_ERR_INVALID_ARGUMENT, "NULL argument");
  const Codebook& cb = codebook();
  std::memcpy(levels8, cb.level, sizeof cb.level);
  std::memcpy(thresholds7, cb.thr, sizeof cb.thr);
  return MKV_OK;
}

mkv_status mkv_plan_decode_multi(mkv_pool* p, int32_t n, const int32_t* ids, int32_t nq, int32_t* chunks, int32_t cap,
                                 int32_t* n_chunks) {
  if (!p || !n_chunks) return fail(MKV_ERR_INVALID_ARGUMENT, "NULL argument");
  mkv_status st = check_batch(p, n, ids, true);
  if (st != MKV_OK) return st;
  if ((st = check_queries(p, n, ids, nq)) != MKV_OK) return st;
  if ((st = build_plan(p, n, ids, nq, false, nullptr)) != MKV_OK) return st;
  p->plan_gen = 0;   // the device copy (if any) no longer matches
  const int nc = int(p->plan_debug.size() / kPlanRecord);
  *n_chunks = nc;
  if (chunks) {
    if (cap < nc) return fail(MKV_ERR_INVALID_ARGUMENT, "cap %d < %d chunks", cap, nc);
    std::memcpy(chunks, p->plan_debug.data(), p->plan_debug.size() * sizeof(int32_t));
  }
  return MKV_OK;
}

mkv_status mkv_plan_decode(mkv_pool* p, int32_t n, const int32_t* ids, int32_t* chunks, int32_t cap, int32_t* n_chunks) {
  return mkv_plan_decode_multi(p, n, ids, 1, chunks, cap, n_chunks);
}

mkv_status mkv_selftest_wait_timeout(mkv_pool* p, int64_t limit_cycles, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (limit_cycles < 1 || limit_cycles > 4000000000LL)
    return fail(MKV_ERR_INVALID_ARGUMENT, "limit_cycles %lld outside [1, 4e9]", static_cast<long long>(limit_cycles));
  if (p->host_only) return fail(MKV_ERR_UNSUPPORTED, "host-only pool: no device error word");
  const cudaError_t e = launch_wait_probe(p->err, limit_cycles, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
  return MKV_OK;
}

mkv_status mkv_inject_plan_slot(mkv_pool* p, int32_t entry, int32_t slot, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (p->host_only) return fail(MKV_ERR_UNSUPPORTED, "host-only pool: no device plan");
  if (p->plan_gen != p->generation || p->plan_gen == 0)
    return fail(MKV_ERR_INVALID_STATE, "no current device plan (decode a batch first)");
  if (entry < 0 || entry >= p->plan_entries)
    return fail(MKV_ERR_INVALID_ARGUMENT, "entry %d outside the plan's %d", entry, p->plan_entries);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const PlanLayout L = plan_layout(p->entry_cap, p->chunk_cap, effective_batch(p->cfg), p->cfg.num_kv_heads);
  uint8_t* dst = p->plan_region + L.entries + size_t(entry) * sizeof(PageEntry) + offsetof(PageEntry, slot);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(dst, &slot, sizeof slot, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "plan entry write");
  p->plan_injected = true;
  return MKV_OK;
}

mkv_status mkv_set_timing_events(mkv_pool* p, void* start, void* stop) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  p->t_start = static_cast<cudaEvent_t>(start);
  p->t_stop = static_cast<cudaEvent_t>(stop);
  return MKV_OK;
}

mkv_status mkv_check_device_errors(mkv_pool* p, mkv_stream_t stream) {
  if (!p) return fail(MKV_ERR_INVALID_ARGUMENT, "pool is NULL");
  if (p->host_only) return MKV_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, p->err, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "error word read");
  if (h) {
    e = cudaMemsetAsync(p->err, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return fail(MKV_ERR_DEVICE_CHECK, "device error word 0x%x (%s%s)", h, (h & kErrWaitTimeout) ? "wait timeout " : "",
                (h & kErrBadPlan) ? "bad plan entry" : "");
  }
  return MKV_OK;
}

}  // extern "C"
