// C ABI of libdflash: handle, validation, device-memory layout, work planning,
// the order of launches of encode / inject / step / accept, and graph capture.
#include "../../include/dflash.h"
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <new>
#include <vector>

using namespace dflash;

namespace {

constexpr int kPlanSMs = 152;        // GB300: 2 dies x 76 SMs
constexpr int kCtasPerSm = 2;        // projection CTAs resident per SM (registers bound it)
// largest ring slice (all sequences of one layer) prefetched into L2 ahead of attention
constexpr size_t kRingPrefetchMax = 32u << 20;
constexpr int kGemmGrid = kPlanSMs * kCtasPerSm;
constexpr int kXkMax = kGemmXkMax;   // activation stage width of the register-fed kernel
// launch timestamp slots of one profiled step (5 launches per layer + 3)
constexpr int kStampSlots = 5 * DFLASH_MAX_LAYERS + 8;
constexpr size_t kAlign = 256;
// largest weight matrix the attention kernel prefetches into L2 (half of L2)
constexpr size_t kAttnPrefetchMax = (size_t)64 << 20;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int cdiv(int a, int b) { return (a + b - 1) / b; }

int wtype_of(int dtype) {
  return dtype == DFLASH_DTYPE_F32 ? W_F32 : dtype == DFLASH_DTYPE_BF16 ? W_BF16
         : dtype == DFLASH_DTYPE_FP8_E4M3 ? W_FP8 : W_FP4;
}
int chunk_of(int wt) { return wt == W_FP8 ? 64 : 32; }

struct Plan {
  int n_tiles = 0, n_mb = 1, cpt = 0, grid = 0, xk = 0;
};

// Stream-K plan of one projection launch: one resident wave of CTAs sharing
// n_tiles x n_mb x (K / kc) chunk units equally.
Plan plan_gemm(int n_tiles, int K, int kc, int n_mb) {
  Plan p;
  p.n_tiles = n_tiles;
  p.n_mb = n_mb;
  p.cpt = cdiv(K, kc);
  const long long units = (long long)n_tiles * n_mb * p.cpt;
  p.grid = (int)std::min<long long>(kGemmGrid, units);
  p.xk = std::min(p.cpt * kc, (kXkMax / kc) * kc);
  return p;
}

struct Geometry {
  int d, qd, kvd, hd, F, V, L, W, Hq, Hkv, fdim, max_seq, max_inject, M_max;
  int wt, kc, dense_bf16, ring_bf16;
};

// The 16-bit activation pair of the projections of a step (or an injection)
// of M rows: fp16 where the products run in fp16 - FP4 weights, and E4M3
// weights below 128 rows (exact in fp16); bf16 otherwise (the tcgen05 kernel
// runs E4M3 batches in bf16).
inline int pair_f16_of(const Geometry& g, int M) { return g.wt == W_FP4 || (g.wt == W_FP8 && M < 128); }

// Bytes of one [rows][K] projection weight buffer (FP4: codes, then block scales).
inline size_t weight_bytes(int wt, int rows, int K) {
  const size_t n = (size_t)rows * K;
  switch (wt) {
    case W_F32: return 4 * n;
    case W_FP8: return n;
    case W_FP4: return n / 2 + n / 16;
    default: return 2 * n;
  }
}

Geometry geometry(const dflash_config& c) {
  Geometry g;
  g.d = c.n_embd;
  g.hd = c.head_dim;
  g.Hq = c.n_head;
  g.Hkv = c.n_head_kv;
  g.qd = c.n_head * c.head_dim;
  g.kvd = c.n_head_kv * c.head_dim;
  g.F = c.n_ff;
  g.V = c.n_vocab;
  g.L = c.n_layer;
  g.W = c.window;
  g.fdim = c.n_target_layers * c.target_embd;
  g.max_seq = c.max_seq;
  g.max_inject = c.max_inject;
  g.M_max = c.max_seq * DFLASH_BLOCK;
  g.wt = wtype_of(c.weight_dtype);
  g.kc = chunk_of(g.wt);
  g.dense_bf16 = c.dense_dtype == DFLASH_DTYPE_BF16;
  g.ring_bf16 = c.ring_dtype == DFLASH_DTYPE_BF16;
  return g;
}

// the projection launches of one step / inject, as (tiles, K, chunk width)
struct GemmShape {
  int n_tiles, K, kc;
};

void step_shapes(const Geometry& g, GemmShape out[5]) {
  const int kc = tma_chunk_k(g.wt);
  out[0] = {cdiv(g.qd + 2 * g.kvd, kTileRows), g.d, kc};   // q/k/v
  out[1] = {cdiv(g.d, kTileRows), g.qd, kc};               // o
  out[2] = {cdiv(g.F, kTileRows / 2), g.d, kc};            // gate/up
  out[3] = {cdiv(g.d, kTileRows), g.F, kc};                // down
  out[4] = {cdiv(g.V, kTileRows), g.d, kc};                // lm head
}

void inject_shapes(const Geometry& g, GemmShape out[2]) {
  const int dense_kc = 32;
  out[0] = {cdiv(g.d, kTileRows), g.fdim, dense_kc};               // fc
  out[1] = {cdiv(2 * g.L * g.kvd, kTileRows), g.d, g.kc};          // all-layer wk/wv
}

struct Layout {
  size_t status, inv_freq, counters, h, ss, qbuf, kblk, vblk, rope_step, am_part;
  size_t xn_hi, xn_lo, attn_hi, attn_lo, act_hi, act_lo;
  size_t logits_int, drafts_int, idl_int, npast_int, partial;
  size_t inj_raw, inj_ss, inj_rope, inj_hi, inj_lo, loop_pos, loop_cnt, loop_H, stamps;
  size_t attn_part, attn_ml, attn_cnt, chain_partial, chain_cnt, chain_item, chain_mb, chain_done;
  size_t plan_nv, plan_sub;
  size_t total;
  int attn_groups, chain_item_stride;
  size_t partial_floats;
  int n_counters, ss_parts, ss_ld, lm_tiles;
  size_t ring_seq_bytes, ring_kv_bytes, ring_total;
};

Layout layout(const dflash_config& c) {
  const Geometry g = geometry(c);
  Layout L{};
  GemmShape ss_[5], is_[2];
  step_shapes(g, ss_);
  inject_shapes(g, is_);
  // two partial tiles per CTA of the stream-K grid; one ticket per output tile
  const size_t partial = (size_t)2 * kGemmGrid * 16 * kTileRows;
  int counters = 0;
  for (auto& s : ss_) counters = std::max(counters, g.max_seq * s.n_tiles);
  for (auto& s : is_) counters = std::max(counters, cdiv(g.max_inject, 16) * s.n_tiles);
  L.partial_floats = partial;
  L.n_counters = counters + g.max_seq;    // + the logits-argmax tickets (one per 16-row block)
  L.ss_parts = cdiv(g.d, kTileRows);
  L.ss_ld = std::max(g.M_max, g.max_inject);
  L.lm_tiles = ss_[4].n_tiles;

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  L.status = take(sizeof(unsigned));
  L.inv_freq = take(sizeof(double) * (g.hd / 2));
  L.counters = take(sizeof(int) * L.n_counters);
  L.h = take(sizeof(float) * g.M_max * g.d);
  L.ss = take(sizeof(float) * (size_t)L.ss_parts * L.ss_ld);
  L.qbuf = take(sizeof(float) * g.M_max * g.qd);
  L.kblk = take(sizeof(float) * g.M_max * g.kvd);
  L.vblk = take(sizeof(float) * g.M_max * g.kvd);
  L.xn_hi = take(sizeof(uint16_t) * (size_t)g.M_max * g.d);
  L.xn_lo = take(sizeof(uint16_t) * (size_t)g.M_max * g.d);
  L.attn_hi = take(sizeof(uint16_t) * (size_t)g.M_max * g.qd);
  L.attn_lo = take(sizeof(uint16_t) * (size_t)g.M_max * g.qd);
  L.act_hi = take(sizeof(uint16_t) * (size_t)g.M_max * g.F);
  L.act_lo = take(sizeof(uint16_t) * (size_t)g.M_max * g.F);
  L.rope_step = take(sizeof(float2) * g.M_max * (g.hd / 2));
  L.am_part = take(sizeof(float2) * (size_t)L.lm_tiles * g.M_max);
  L.logits_int = take(sizeof(float) * (size_t)g.M_max * g.V);
  L.drafts_int = take(sizeof(int32_t) * g.max_seq * (DFLASH_BLOCK - 1));
  L.idl_int = take(sizeof(int32_t) * g.max_seq);
  L.npast_int = take(sizeof(int32_t) * g.max_seq);
  L.partial = take(sizeof(float) * std::max<size_t>(partial, 1));
  L.inj_raw = take(sizeof(float) * (size_t)g.max_inject * g.d);
  L.inj_ss = take(sizeof(float) * (size_t)L.ss_parts * L.ss_ld);
  L.inj_rope = take(sizeof(float2) * (size_t)g.max_inject * (g.hd / 2));
  // H_t as a bf16 hi/lo pair for injections of >= 128 rows on the tcgen05 path
  // (and for every injection with FP4 weights, which runs on the 16-row TMA kernel)
  const bool inj_pair = (g.max_inject >= 128 && (g.wt == W_BF16 || g.wt == W_FP8)) || g.wt == W_FP4;
  L.inj_hi = take(inj_pair ? sizeof(uint16_t) * (size_t)std::max(g.max_inject, 1) * g.d : 0);
  L.inj_lo = take(inj_pair ? sizeof(uint16_t) * (size_t)std::max(g.max_inject, 1) * g.d : 0);
  // speculative-loop turn: block positions, accepted-row counts, encoded rows
  L.loop_pos = take(sizeof(int32_t) * (size_t)g.max_seq * DFLASH_BLOCK);
  L.loop_cnt = take(sizeof(int32_t) * (size_t)g.max_seq);
  L.loop_H = take(sizeof(float) * (size_t)g.max_seq * DFLASH_BLOCK * g.d);
  L.stamps = take(sizeof(unsigned long long) * 2 * kStampSlots);
  // split-window attention: partial rows of its largest grid, and two counters
  // per (sequence, kv head, query head) - at least one per head group
  L.attn_part = take(sizeof(float) * (size_t)kAttnSplitMaxCtas * kAttnPartFloats);
  L.attn_ml = take(sizeof(float2) * (size_t)kAttnSplitMaxCtas * 64);
  L.attn_groups = g.max_seq * g.Hq;
  L.attn_cnt = take(sizeof(int) * 2 * (size_t)L.attn_groups);
  // stream-K attention plan: listed sub-chunks of each sequence
  L.plan_nv = take(sizeof(int) * (size_t)g.max_seq);
  L.plan_sub = take(sizeof(int) * (size_t)g.max_seq * 64);
  // projection chains: per phase its partial tiles and tickets, item flags and
  // per-block counts; one chain counter
  L.chain_partial = take(sizeof(float) * (size_t)kChainMax * 2 * kGemmGrid * 16 * kTileRows);
  L.chain_cnt = take(sizeof(int) * (size_t)kChainMax * L.n_counters);
  int items = 0;
  for (auto& s : ss_) items = std::max(items, g.max_seq * s.n_tiles);
  L.chain_item_stride = items;
  L.chain_item = take(sizeof(int) * (size_t)kChainMax * items);
  L.chain_mb = take(sizeof(int) * (size_t)kChainMax * g.max_seq);
  L.chain_done = take(sizeof(int));
  L.total = off;

  L.ring_kv_bytes = (size_t)g.L * 2 * g.Hkv * g.W * g.hd * (g.ring_bf16 ? 2 : 4);
  L.ring_seq_bytes = L.ring_kv_bytes;
  L.ring_total = align_up(L.ring_kv_bytes * g.max_seq) + sizeof(int32_t) * (size_t)g.max_seq * g.W;
  return L;
}

int validate(const dflash_config* c) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  if (c->n_layer < 1 || c->n_embd < 1 || c->n_head < 1 || c->n_head_kv < 1 || c->head_dim < 1 ||
      c->n_ff < 1 || c->window < 1 || c->n_vocab < 1 || c->n_target_layers < 1 ||
      c->target_embd < 1 || c->max_seq < 1 || c->max_inject < 0)
    return DFLASH_ERR_INVALID_ARG;
  if (c->mask_token_id < 0 || c->mask_token_id >= c->n_vocab) return DFLASH_ERR_INVALID_ARG;
  if (!(c->eps >= 0.f) || !(c->rope_theta > 0.0)) return DFLASH_ERR_INVALID_ARG;
  if (c->weight_dtype < DFLASH_DTYPE_F32 || c->weight_dtype > DFLASH_DTYPE_FP4_E2M1)
    return DFLASH_ERR_INVALID_ARG;
  if ((c->dense_dtype != DFLASH_DTYPE_F32 && c->dense_dtype != DFLASH_DTYPE_BF16) ||
      (c->ring_dtype != DFLASH_DTYPE_F32 && c->ring_dtype != DFLASH_DTYPE_BF16))
    return DFLASH_ERR_UNSUPPORTED;
  if (c->n_layer > DFLASH_MAX_LAYERS) return DFLASH_ERR_UNSUPPORTED;
  if (c->n_head % c->n_head_kv) return DFLASH_ERR_UNSUPPORTED;
  if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128) return DFLASH_ERR_UNSUPPORTED;
  const int kc = c->weight_dtype == DFLASH_DTYPE_FP4_E2M1 ? 256
                 : c->weight_dtype == DFLASH_DTYPE_FP8_E4M3 ? 64 : 32;
  const int qd = c->n_head * c->head_dim;
  if (c->n_embd % kc || qd % kc || c->n_ff % kc) return DFLASH_ERR_UNSUPPORTED;
  if ((c->n_target_layers * c->target_embd) % 32) return DFLASH_ERR_UNSUPPORTED;
  // one warp per query head of a kv group in the attention CTA
  if (c->n_head / c->n_head_kv > 8) return DFLASH_ERR_UNSUPPORTED;
  // the attention CTA's staging must fit one SM's shared memory (227 KB per block,
  // 1 KB kept for its static barriers)
  if (attn_cluster_smem(c->n_head / c->n_head_kv, c->head_dim, c->ring_dtype == DFLASH_DTYPE_F32) >
          232448 - 1024 ||
      attn_split_smem(c->n_head / c->n_head_kv, c->head_dim, c->ring_dtype == DFLASH_DTYPE_F32) >
          232448 - 1024)
    return DFLASH_ERR_UNSUPPORTED;
  return DFLASH_OK;
}

}  // namespace

struct dflash_handle {
  dflash_config cfg;
  dflash_weights w;
  Geometry g;
  Layout L;
  char* ring;
  char* scratch;
  // tensor maps of the step's weights (wq, wk, wv, wo, gate, up, down per layer,
  // the LM head) and of the three activation-pair buffers
  CUtensorMap tm_layer[DFLASH_MAX_LAYERS][7];
  CUtensorMap tm_lm;
  // bf16 / E4M3 weights in 64-row boxes for the 16-row kernel
  CUtensorMap tm_layer64[DFLASH_MAX_LAYERS][7];
  CUtensorMap tm_lm64;
  // FP4: block scales as [groups of 16 rows][K bytes], 256 x 4 boxes
  CUtensorMap tm_scale64[DFLASH_MAX_LAYERS][7];
  CUtensorMap tm_lm_s64;
  CUtensorMap tm_xn[2], tm_attn[2], tm_act[2];
  // FP4: the same pairs as 4-D hi+lo maps (all three, then the injection pair)
  CUtensorMap tm_x4[4];
  bool x4 = false;
  // the same for the tcgen05 kernel (128-row activation boxes, 32-row weight boxes)
  bool dense = false;
  CUtensorMap td_layer[DFLASH_MAX_LAYERS][7];
  CUtensorMap td_lm;
  CUtensorMap td_xn[2], td_attn[2], td_act[2];
  // FP4: the injection input pair for the 16-row kernel
  CUtensorMap tm_inj[2];
  // bf16 ring with hd >= 64: the attention kernel's staging map
  CUtensorMap tm_ring;
  // prefill on the tcgen05 path (>= 128 rows): fc (bf16 features), all-layer
  // wk / wv, and the injection input pair
  bool enc_dense = false, inj_dense = false;
  CUtensorMap td_fc;
  CUtensorMap td_kv[DFLASH_MAX_LAYERS][2];
  CUtensorMap td_inj[2];
  cudaStream_t cap_stream = nullptr;
  // captured graphs, one per block width (a capture bakes its row count): the
  // step (+ accept) of dflash_capture and the loop turn of dflash_capture_loop
  cudaGraph_t graphs[DFLASH_BLOCK + 1] = {};
  cudaGraphExec_t execs[DFLASH_BLOCK + 1] = {};
  cudaGraph_t loop_graphs[DFLASH_BLOCK + 1] = {};
  cudaGraphExec_t loop_execs[DFLASH_BLOCK + 1] = {};
  int width = DFLASH_BLOCK;   // block rows of step / accept / advance / capture
  char err[512];
  // 16-row steps may chain their projections (o, gate/up, down, next q/k/v) per
  // layer (dflash_set_chain) when the device holds the chain's grid at once (chain_ok)
  bool chain = false, chain_ok = false;
  // launch-class profiling: events around eager calls (prof), or device
  // timestamps of every step launch, eager or captured (stamps)
  bool prof = false;
  bool stamps = false;
  std::vector<int> stamp_cls;   // class of each timestamp slot of the last recorded step
  bool capturing = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  struct Rec { int cls; cudaEvent_t a, b; };
  std::vector<Rec> recs;
  int open_cls = -1;
  cudaEvent_t open_ev = nullptr;

  template <typename T>
  T* S(size_t off) const { return reinterpret_cast<T*>(scratch + off); }
  unsigned* status() const { return S<unsigned>(L.status); }
  int32_t* ring_pos(int seq) const {
    return reinterpret_cast<int32_t*>(ring + align_up(L.ring_kv_bytes * g.max_seq)) + (size_t)seq * g.W;
  }
  char* ring_seq(int seq) const { return ring + (size_t)seq * L.ring_seq_bytes; }
};

namespace {

int cuda_fail(dflash_handle* h, cudaError_t e, const char* where) {
  if (h) std::snprintf(h->err, sizeof(h->err), "%s: %s", where, cudaGetErrorString(e));
  return DFLASH_ERR_CUDA;
}

// The runtime's last-error slot is shared with every other user of CUDA in the
// process; clear it on entry so a stale error is not reported as this call's.
inline void clear_stale_error() { (void)cudaGetLastError(); }

#define DF_CHECK(h, call)                                   \
  do {                                                      \
    cudaError_t e_ = (call);                                \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, #call);  \
  } while (0)

// cuTensorMapEncodeTiled through the runtime's driver entry point (the library
// does not link libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// 2-D map of a row-major [rows][cols] matrix with boxes of box_cols x box_rows
// elements; out-of-range rows / columns read as zero.
bool make_map(CUtensorMap* m, const void* base, int wt, uint64_t cols, uint64_t rows,
              uint32_t box_cols, uint32_t box_rows, bool swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType dt = wt == W_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : wt == W_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t esz = wt == W_F32 ? 4 : wt == W_BF16 ? 2 : 1;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esz};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 16-row x 128-byte swizzled boxes (the 16-row TMA kernel)
bool make_map(CUtensorMap* m, const void* base, int wt, uint64_t cols, uint64_t rows) {
  const uint32_t esz = wt == W_F32 ? 4 : wt == W_BF16 ? 2 : 1;
  return make_map(m, base, wt, cols, rows, 128 / esz, 16, true);
}

enum ProfClass {
  PC_EMBED = 0, PC_QKV, PC_ATTN, PC_MERGE, PC_O, PC_GATEUP, PC_DOWN, PC_LM, PC_ENCODE, PC_INJECT,
  PC_ACCEPT, PC_CHAIN
};

cudaEvent_t prof_event(dflash_handle* h) {
  if (h->ev_used == h->ev_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    h->ev_pool.push_back(e);
  }
  return h->ev_pool[h->ev_used++];
}

// bracket the launches of one class with events on the launching stream
void prof_begin(dflash_handle* h, int cls, cudaStream_t st) {
  if (!h->prof || h->capturing) return;
  h->open_ev = prof_event(h);
  h->open_cls = cls;
  if (h->open_ev) cudaEventRecord(h->open_ev, st);
}

void prof_end(dflash_handle* h, cudaStream_t st) {
  if (!h->prof || h->capturing || !h->open_ev) return;
  cudaEvent_t b = prof_event(h);
  if (!b) return;
  cudaEventRecord(b, st);
  h->recs.push_back({h->open_cls, h->open_ev, b});
  h->open_ev = nullptr;
}

// The next launch timestamp slot (class `cls`), or null when stamps are off.
unsigned long long* stamp_slot(dflash_handle* h, int cls) {
  if (!h->stamps || (int)h->stamp_cls.size() >= kStampSlots) return nullptr;
  unsigned long long* s = h->S<unsigned long long>(h->L.stamps) + 2 * h->stamp_cls.size();
  h->stamp_cls.push_back(cls);
  return s;
}

// Start a new stamp record: every slot zeroed on the stream ahead of the step.
cudaError_t stamp_reset(dflash_handle* h, cudaStream_t st) {
  h->stamp_cls.clear();
  if (!h->stamps) return cudaSuccess;
  return cudaMemsetAsync(h->scratch + h->L.stamps, 0, sizeof(unsigned long long) * 2 * kStampSlots, st);
}

#define PROF(h, cls, st, call)     \
  do {                             \
    prof_begin(h, cls, st);        \
    DF_CHECK(h, call);             \
    prof_end(h, st);               \
  } while (0)

GemmParams base_params(const dflash_handle* h) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.eps = h->cfg.eps;
  p.rms_len = h->g.d;
  p.norm_bf16 = h->g.dense_bf16;
  p.partial = h->S<float>(h->L.partial);
  p.counters = h->S<int>(h->L.counters);
  p.status = h->status();
  p.hd = h->g.hd;
  p.qd = h->g.qd;
  p.kvd = h->g.kvd;
  p.window = h->g.W;
  p.n_head_kv = h->g.Hkv;
  p.ring_bf16 = h->g.ring_bf16;
  // FP4 weights multiply in fp16: their projections' activation pairs are fp16
  p.pair_f16 = h->g.wt == W_FP4;   // the step sets its own (pair_f16_of)
  return p;
}

void set_plan(GemmParams& p, const GemmShape& s, int n_mb) {
  const Plan pl = plan_gemm(s.n_tiles, s.K, s.kc, n_mb);
  p.n_tiles = pl.n_tiles;
  p.n_mb = pl.n_mb;
  p.cpt = pl.cpt;
  p.grid = pl.grid;
  p.xk = pl.xk;
  p.K = s.K;
}

// Projection launch on the TMA kernel: X is one of the activation-pair buffers.
void set_tma_inputs(GemmParams& p, const CUtensorMap* x) {
  p.tm_xh = x[0];
  p.tm_xl = x[1];
  p.has_lo = 1;
  p.x_mode = X_BF16;
}

// Bind a step projection to its tensor maps: the tcgen05 kernel's for >= 128
// activation rows (its own maps, 64-wide k chunks), else the 16-row kernels'.
// Weight maps: layer l, matrices wi[0..nw) (l < 0: the LM head); activations:
// pair xi (0 xn, 1 attn, 2 act).  launch_bound launches it on its kernel.
enum { XP_XN = 0, XP_ATTN = 1, XP_ACT = 2 };

void bind_projection(const dflash_handle* h, GemmParams& p, int l, std::initializer_list<int> wi,
                     int xi) {
  const bool dense = h->dense && p.M >= 128;
  const CUtensorMap* xs[3] = {dense ? h->td_xn : h->tm_xn, dense ? h->td_attn : h->tm_attn,
                              dense ? h->td_act : h->tm_act};
  set_tma_inputs(p, xs[xi]);
  if (h->x4) {
    p.tm_x4 = h->tm_x4[xi];
    p.x4 = 1;
  }
  int i = 0;
  for (int w : wi) {
    p.tm_w64[i] = l < 0 ? h->tm_lm64 : h->tm_layer64[l][w];
    if (h->g.wt == W_FP4) p.tm_s64[i] = l < 0 ? h->tm_lm_s64 : h->tm_scale64[l][w];
    p.tm_w[i++] = l < 0 ? (dense ? h->td_lm : h->tm_lm)
                        : (dense ? h->td_layer[l][w] : h->tm_layer[l][w]);
  }
  p.w64 = h->g.wt == W_BF16 || h->g.wt == W_FP8 || h->g.wt == W_FP4;
  if (dense) p.cpt = cdiv(p.K, 64);
}

cudaError_t launch_bound(const dflash_handle* h, GemmParams& p, cudaStream_t st) {
  const bool dense = h->dense && p.M >= 128;
  if (h->g.wt == W_FP4) return launch_gemm_fp4(W_FP4, p, st);
  // 16-row E4M3 projections of at least 64 M weights whose k is a multiple of
  // 256 run on the same tensor-memory pipeline (units of 128 rows x 256 k):
  // it streams E4M3 faster than the 16-row TMA kernel's mma.sync path, whose
  // shorter start wins below that (measured on the real drafter's projections)
  if (h->g.wt == W_FP8 && !dense && p.K % 256 == 0 && p.has_lo && (long long)p.N * p.K >= (64ll << 20)) {
    p.cpt = p.K / 256;
    return launch_gemm_fp4(W_FP8, p, st);
  }
  if (!dense) return launch_gemm_tma(h->g.wt, p, st);
  return launch_gemm_umma(h->g.wt, p, st);
}

// the embedding kernel's blocks per row (each writes one partial sum of squares)
int embed_parts(const Geometry& g, const Layout& L) {
  int parts = std::min(4, L.ss_parts);
  while (parts > 1 && g.d % (8 * parts) != 0) --parts;
  return parts;
}

int run_step(dflash_handle* h, int n_seq, const int32_t* id_last, const int32_t* n_past,
             float* logits, int32_t* drafts, cudaStream_t st) {
  clear_stale_error();
  const Geometry& g = h->g;
  const Layout& L = h->L;
  const int M = n_seq * DFLASH_BLOCK;
  GemmShape sh[5];
  step_shapes(g, sh);
  float* hbuf = h->S<float>(L.h);
  float* ss = h->S<float>(L.ss);
  float2* rope = h->S<float2>(L.rope_step);
  uint16_t* xn_hi = h->S<uint16_t>(L.xn_hi);
  uint16_t* xn_lo = h->S<uint16_t>(L.xn_lo);
  DF_CHECK(h, stamp_reset(h, st));
  // h = embeddings; xn = split(h * attn_norm_0); ss = row sums of squares
  PROF(h, PC_EMBED, st, launch_embed(h->w.tok_embd, g.dense_bf16, g.d, g.V, h->cfg.mask_token_id,
                                     id_last, n_past, n_seq, h->S<double>(L.inv_freq), g.hd, hbuf, ss,
                                     rope, h->w.layers[0].attn_norm, xn_hi, xn_lo, pair_f16_of(g, M),
                                     embed_parts(g, L), L.ss_ld, h->status(),
                                     stamp_slot(h, PC_EMBED), st));
  // The projections' parameters (weights, schedule, row statistics, epilogue),
  // bound to their tensor maps by bind_projection.
  // q/k/v of RMSNorm(h) (the 1/rms row scale after the product), per-head q/k
  // norm + rope; n_ss partial sums of squares per row in ss
  auto qkv_p = [&](int l, int n_ss) {
    const dflash_layer_weights& lw = h->w.layers[l];
    GemmParams p = base_params(h);
    p.pair_f16 = pair_f16_of(g, M);
    set_plan(p, sh[0], n_seq);
    p.M = M;
    p.ss = ss; p.n_ss = n_ss; p.ss_ld = L.ss_ld; p.row_scale = 1;
    p.seg[0] = {lw.wq, lw.wq_scale, 0, g.qd};
    p.seg[1] = {lw.wk, lw.wk_scale, g.qd, g.kvd};
    p.seg[2] = {lw.wv, lw.wv_scale, g.qd + g.kvd, g.kvd};
    p.nseg = 3; p.N = g.qd + 2 * g.kvd; p.map = MAP_SEGMENTS;
    p.epi = EPI_QKV; p.out = h->S<float>(L.qbuf); p.ldo = g.qd;
    p.kblk = h->S<float>(L.kblk); p.vblk = h->S<float>(L.vblk);
    p.q_norm = lw.q_norm; p.k_norm = lw.k_norm; p.rope_cs = rope;
    // this layer's ring K/V of every sequence into L2 for the attention kernel
    const size_t layer_bytes = L.ring_kv_bytes / g.L;
    if ((size_t)n_seq * layer_bytes <= kRingPrefetchMax) {
      p.pf_base = h->ring + (size_t)l * layer_bytes;
      p.pf_bytes = layer_bytes;
      p.pf_stride = L.ring_seq_bytes;
      p.pf_count = n_seq;
    }
    bind_projection(h, p, l, {0, 1, 2}, XP_XN);
    return p;
  };
  // o projection + residual; next input xn = split(h * ffn_norm)
  auto o_p = [&](int l) {
    GemmParams p = base_params(h);
    p.pair_f16 = pair_f16_of(g, M);
    set_plan(p, sh[1], n_seq);
    p.M = M;
    p.seg[0] = {h->w.layers[l].wo, h->w.layers[l].wo_scale, 0, g.d};
    p.nseg = 1; p.N = g.d; p.map = MAP_SEGMENTS;
    p.epi = EPI_RESID_SS; p.out = hbuf; p.ldo = g.d; p.ss_out = ss; p.ss_out_ld = L.ss_ld;
    p.pair_hi = xn_hi; p.pair_lo = xn_lo; p.pair_ld = g.d; p.pair_norm = h->w.layers[l].ffn_norm;
    bind_projection(h, p, l, {3}, XP_ATTN);
    return p;
  };
  // gate/up of RMSNorm(h) + SwiGLU -> act pair
  auto gu_p = [&](int l) {
    const dflash_layer_weights& lw = h->w.layers[l];
    GemmParams p = base_params(h);
    p.pair_f16 = pair_f16_of(g, M);
    set_plan(p, sh[2], n_seq);
    p.M = M;
    p.ss = ss; p.n_ss = sh[1].n_tiles; p.ss_ld = L.ss_ld; p.row_scale = 1;
    p.seg[0] = {lw.gate, lw.gate_scale, 0, g.F};
    p.seg[1] = {lw.up, lw.up_scale, 0, g.F};
    p.nseg = 2; p.N = 2 * g.F; p.map = MAP_SWIGLU;
    p.epi = EPI_SWIGLU; p.out = nullptr;
    p.pair_hi = h->S<uint16_t>(L.act_hi); p.pair_lo = h->S<uint16_t>(L.act_lo); p.pair_ld = g.F;
    bind_projection(h, p, l, {4, 5}, XP_XN);
    return p;
  };
  // down projection + residual; next input xn = split(h * next norm)
  auto down_p = [&](int l) {
    GemmParams p = base_params(h);
    p.pair_f16 = pair_f16_of(g, M);
    set_plan(p, sh[3], n_seq);
    p.M = M;
    p.seg[0] = {h->w.layers[l].down, h->w.layers[l].down_scale, 0, g.d};
    p.nseg = 1; p.N = g.d; p.map = MAP_SEGMENTS;
    p.epi = EPI_RESID_SS; p.out = hbuf; p.ldo = g.d; p.ss_out = ss; p.ss_out_ld = L.ss_ld;
    p.pair_hi = xn_hi; p.pair_lo = xn_lo; p.pair_ld = g.d;
    p.pair_norm = l + 1 < g.L ? h->w.layers[l + 1].attn_norm : h->w.out_norm;
    bind_projection(h, p, l, {6}, XP_ACT);
    return p;
  };
  // LM head of RMSNorm(h) (out_norm folded into xn by the last down projection)
  auto lm_p = [&]() {
    GemmParams p = base_params(h);
    p.pair_f16 = pair_f16_of(g, M);
    set_plan(p, sh[4], n_seq);
    p.M = M;
    p.ss = ss; p.n_ss = sh[3].n_tiles; p.ss_ld = L.ss_ld; p.row_scale = 1;
    p.seg[0] = {h->w.lm_head, h->w.lm_head_scale, 0, g.V};
    p.nseg = 1; p.N = g.V; p.map = MAP_SEGMENTS;
    p.epi = EPI_LOGITS; p.out = logits; p.ldo = g.V;
    p.am_part = h->S<float2>(L.am_part);
    p.am_counter = h->S<int>(L.counters) + (L.n_counters - g.max_seq);
    p.drafts = drafts;
    p.block_width = h->width;
    bind_projection(h, p, -1, {0}, XP_XN);
    return p;
  };
  auto attn_params = [&](int l) {
    AttnParams a;
    std::memset(&a, 0, sizeof(a));
    a.q = h->S<float>(L.qbuf); a.kblk = h->S<float>(L.kblk); a.vblk = h->S<float>(L.vblk);
    a.ring = h->ring; a.ring_pos = h->ring_pos(0); a.n_past = n_past;
    a.ring_bf16 = g.ring_bf16; a.layer = l; a.n_layer = g.L;
    a.n_head = g.Hq; a.n_head_kv = g.Hkv; a.hd = g.hd; a.window = g.W;
    a.scale = (float)(1.0 / std::sqrt((double)g.hd));
    a.out_hi = h->S<uint16_t>(L.attn_hi); a.out_lo = h->S<uint16_t>(L.attn_lo);
    a.pair_f16 = pair_f16_of(g, M);
    a.tm_ring = h->tm_ring;
    a.status = h->status();
    a.block_width = h->width;
    a.part_o = h->S<float>(L.attn_part);
    a.part_ml = h->S<float2>(L.attn_ml);
    a.counters = h->S<int>(L.attn_cnt);
    a.plan_nv = h->S<int>(L.plan_nv);
    a.plan_sub = h->S<int>(L.plan_sub);
    // the o projection's weights into L2 while attention publishes and merges
    // (measured: real_bf16 969 -> 960 us per step; fp32 weights, 109 MB at the
    // real dimensions, crowd L2 and are not prefetched)
    const size_t o_bytes = weight_bytes(g.wt, g.d, g.qd);
    if (o_bytes <= kAttnPrefetchMax) {
      a.pf_base = static_cast<const char*>(h->w.layers[l].wo);
      a.pf_bytes = o_bytes;
    }
    return a;
  };
  auto attention = [&](int l) -> int {
    AttnParams a = attn_params(l);
    a.stamp = stamp_slot(h, PC_ATTN);
    PROF(h, PC_ATTN, st, launch_attention(a, n_seq, st));
    return DFLASH_OK;
  };
  // the stream-K attention's plan of this step (its ring and positions do not
  // change within the step: one plan serves every layer)
  if (attention_kind(attn_params(0), n_seq) == ATTN_STREAM)
    PROF(h, PC_ATTN, st, launch_attention_plan(attn_params(0), n_seq, st));

  // 16-row blocks with bf16 / fp32 / E4M3 weights: per layer one persistent
  // launch chains o, gate/up, down and the next layer's q/k/v (the LM head
  // after the last layer) between two attention launches
  if (h->chain && M < 128) {
    GemmParams p = qkv_p(0, embed_parts(g, L));
    p.stamp = stamp_slot(h, PC_QKV);
    PROF(h, PC_QKV, st, launch_bound(h, p, st));
    for (int l = 0; l < g.L; ++l) {
      int rc = attention(l);
      if (rc != DFLASH_OK) return rc;
      ChainParams<kChainMax> cp;
      std::memset(&cp, 0, sizeof(cp));
      cp.ph[0] = o_p(l);
      cp.ph[1] = gu_p(l);
      cp.ph[2] = down_p(l);
      cp.ph[3] = l + 1 < g.L ? qkv_p(l + 1, sh[3].n_tiles) : lm_p();
      cp.n_phase = kChainMax;
      for (int k = 0; k < kChainMax; ++k) {
        cp.ph[k].partial = h->S<float>(L.chain_partial) + (size_t)k * 2 * kGemmGrid * 16 * kTileRows;
        cp.ph[k].counters = h->S<int>(L.chain_cnt) + (size_t)k * L.n_counters;
      }
      cp.item_done = h->S<int>(L.chain_item);
      cp.all_done = h->S<int>(L.chain_mb);
      cp.chain_done = h->S<int>(L.chain_done);
      cp.item_stride = L.chain_item_stride;
      cp.mb_stride = g.max_seq;
      cp.ph[0].stamp = stamp_slot(h, PC_CHAIN);
      PROF(h, PC_CHAIN, st, launch_gemm_chain(g.wt, cp, st));
    }
    return DFLASH_OK;
  }

  int n_ss = embed_parts(g, L);
  for (int l = 0; l < g.L; ++l) {
    GemmParams p = qkv_p(l, n_ss);
    p.stamp = stamp_slot(h, PC_QKV);
    PROF(h, PC_QKV, st, launch_bound(h, p, st));
    int rc = attention(l);
    if (rc != DFLASH_OK) return rc;
    p = o_p(l);
    p.stamp = stamp_slot(h, PC_O);
    PROF(h, PC_O, st, launch_bound(h, p, st));
    p = gu_p(l);
    p.stamp = stamp_slot(h, PC_GATEUP);
    PROF(h, PC_GATEUP, st, launch_bound(h, p, st));
    p = down_p(l);
    p.stamp = stamp_slot(h, PC_DOWN);
    PROF(h, PC_DOWN, st, launch_bound(h, p, st));
    n_ss = sh[3].n_tiles;
  }
  GemmParams p = lm_p();
  p.stamp = stamp_slot(h, PC_LM);
  PROF(h, PC_LM, st, launch_bound(h, p, st));
  return DFLASH_OK;
}

// Tensor maps of every weight the step streams and of the activation pairs.
// FP4 matrix [rows][cols]: its code bytes as [rows][cols/2] (16-row x 128-byte
// swizzled boxes); the kernel reads the block scales behind them by bulk copies
bool make_fp4_map(CUtensorMap* codes, const void* base, uint64_t cols, uint64_t rows) {
  return make_map(codes, base, W_FP8, cols / 2, rows, 128, 16, true);
}

// The same codes in 64-row boxes, and the block scales behind them as a 2-D
// byte tensor [ceil(rows/16) groups][cols bytes] in boxes of 256 bytes x 4
// groups (the scales of 64 rows x 256 k)
// An activation pair (hi at `hi`, lo at `lo` > hi, each [rows][cols] bf16-sized
// elements) as one 4-D tensor: dims (64 k, rows, hi|lo, cols/64 k boxes),
// boxes of 64 x 16 x 2 x 4 with the 128-byte swizzle: per 64 k, 16 hi rows then
// 16 lo rows
bool make_pair_map4(CUtensorMap* m, const void* hi, const void* lo, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || lo <= hi) return false;
  const cuuint64_t dims[4] = {64, rows, 2, cols / 64};
  const cuuint64_t strides[3] = {cols * 2,
                                 (cuuint64_t)(static_cast<const char*>(lo) - static_cast<const char*>(hi)),
                                 128};
  const cuuint32_t box[4] = {64, 16, 2, 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(hi), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_fp4_maps64(CUtensorMap* codes, CUtensorMap* scales, const void* base, uint64_t cols,
                     uint64_t rows) {
  const char* b = static_cast<const char*>(base);
  return make_map(codes, b, W_FP8, cols / 2, rows, 128, 64, true) &&
         make_map(scales, b + rows * cols / 2, W_FP8, cols, (rows + 15) / 16, 256, 4, false);
}

bool build_maps(dflash_handle* h) {
  const Geometry& g = h->g;
  const Layout& L = h->L;
  for (int l = 0; l < g.L; ++l) {
    const dflash_layer_weights& w = h->w.layers[l];
    const void* mats[7] = {w.wq, w.wk, w.wv, w.wo, w.gate, w.up, w.down};
    const int rows[7] = {g.qd, g.kvd, g.kvd, g.d, g.F, g.F, g.d};
    const int cols[7] = {g.d, g.d, g.d, g.qd, g.d, g.d, g.F};
    for (int i = 0; i < 7; ++i) {
      const bool ok = g.wt == W_FP4 ? make_fp4_map(&h->tm_layer[l][i], mats[i], cols[i], rows[i])
                                    : make_map(&h->tm_layer[l][i], mats[i], g.wt, cols[i], rows[i]);
      if (!ok) return false;
      if ((g.wt == W_BF16 || g.wt == W_FP8) &&
          !make_map(&h->tm_layer64[l][i], mats[i], g.wt, cols[i], rows[i], g.wt == W_BF16 ? 64 : 128, 64, true))
        return false;
      if (g.wt == W_FP4 && !make_fp4_maps64(&h->tm_layer64[l][i], &h->tm_scale64[l][i], mats[i], cols[i], rows[i]))
        return false;
    }
  }
  if (g.wt == W_FP4 ? !make_fp4_map(&h->tm_lm, h->w.lm_head, g.d, g.V)
                    : !make_map(&h->tm_lm, h->w.lm_head, g.wt, g.d, g.V))
    return false;
  if ((g.wt == W_BF16 || g.wt == W_FP8) &&
      !make_map(&h->tm_lm64, h->w.lm_head, g.wt, g.d, g.V, g.wt == W_BF16 ? 64 : 128, 64, true))
    return false;
  if (g.wt == W_FP4 && !make_fp4_maps64(&h->tm_lm64, &h->tm_lm_s64, h->w.lm_head, g.d, g.V)) return false;
  const size_t pairs[3][2] = {{L.xn_hi, L.xn_lo}, {L.attn_hi, L.attn_lo}, {L.act_hi, L.act_lo}};
  const int kdim[3] = {g.d, g.qd, g.F};
  CUtensorMap* dst[3] = {h->tm_xn, h->tm_attn, h->tm_act};
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 2; ++j)
      if (!make_map(&dst[i][j], h->scratch + pairs[i][j], W_BF16, kdim[i], g.M_max)) return false;
  // prefill on the tcgen05 path: encode when features and fc are bf16, injection
  // when the weights are bf16 or E4M3, for calls of >= 128 rows
  h->enc_dense = g.max_inject >= 128 && g.dense_bf16;
  if (h->enc_dense && !make_map(&h->td_fc, h->w.fc, W_BF16, g.fdim, g.d, 64, 32, true)) return false;
  h->inj_dense = g.max_inject >= 128 && (g.wt == W_BF16 || g.wt == W_FP8);
  if (h->inj_dense) {
    const bool swk = g.wt == W_BF16;
    for (int l = 0; l < g.L; ++l) {
      if (!make_map(&h->td_kv[l][0], h->w.layers[l].wk, g.wt, g.d, g.kvd, 64, 32, swk)) return false;
      if (!make_map(&h->td_kv[l][1], h->w.layers[l].wv, g.wt, g.d, g.kvd, 64, 32, swk)) return false;
    }
    if (!make_map(&h->td_inj[0], h->scratch + L.inj_hi, W_BF16, g.d, g.max_inject, 64, 128, true) ||
        !make_map(&h->td_inj[1], h->scratch + L.inj_lo, W_BF16, g.d, g.max_inject, 64, 128, true))
      return false;
  }
  if (g.ring_bf16 && g.hd >= 64) {
    const uint64_t rows = (uint64_t)g.max_seq * g.L * 2 * g.Hkv * g.W;
    if (rows >= (1ull << 31) ||
        !make_map(&h->tm_ring, h->ring, W_BF16, g.hd, rows, 64, 64, true))
      return false;
  }
  if (g.wt == W_FP4 || g.wt == W_FP8) {
    // the 4-D pair maps; a driver that refuses them leaves the 2-D path (x4 off)
    h->x4 = true;
    for (int i = 0; i < 3; ++i)
      h->x4 = h->x4 && make_pair_map4(&h->tm_x4[i], h->scratch + pairs[i][0], h->scratch + pairs[i][1],
                                      kdim[i], g.M_max);
    if (g.max_inject > 0)
      h->x4 = h->x4 && make_pair_map4(&h->tm_x4[3], h->scratch + L.inj_hi, h->scratch + L.inj_lo, g.d,
                                      g.max_inject);
  }
  if (g.wt == W_FP4 && g.max_inject > 0 &&
      (!make_map(&h->tm_inj[0], h->scratch + L.inj_hi, W_BF16, g.d, g.max_inject) ||
       !make_map(&h->tm_inj[1], h->scratch + L.inj_lo, W_BF16, g.d, g.max_inject)))
    return false;
  // tcgen05 path: batches of >= 128 activation rows with bf16 or E4M3 weights
  h->dense = g.M_max >= 128 && (g.wt == W_BF16 || g.wt == W_FP8);
  if (!h->dense) return true;
  const bool sw = g.wt == W_BF16;   // raw E4M3 tiles are widened by threads, not read by the MMA
  for (int l = 0; l < g.L; ++l) {
    const dflash_layer_weights& w = h->w.layers[l];
    const void* mats[7] = {w.wq, w.wk, w.wv, w.wo, w.gate, w.up, w.down};
    const int rows[7] = {g.qd, g.kvd, g.kvd, g.d, g.F, g.F, g.d};
    const int cols[7] = {g.d, g.d, g.d, g.qd, g.d, g.d, g.F};
    for (int i = 0; i < 7; ++i)
      if (!make_map(&h->td_layer[l][i], mats[i], g.wt, cols[i], rows[i], 64, 32, sw)) return false;
  }
  if (!make_map(&h->td_lm, h->w.lm_head, g.wt, g.d, g.V, 64, 32, sw)) return false;
  CUtensorMap* ddst[3] = {h->td_xn, h->td_attn, h->td_act};
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 2; ++j)
      if (!make_map(&ddst[i][j], h->scratch + pairs[i][j], W_BF16, kdim[i], g.M_max, 64, 128, true))
        return false;
  return true;
}

bool bad_ptr(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u); }

int check_weights(const dflash_config* c, const dflash_weights* w) {
  if (!w) return DFLASH_ERR_INVALID_ARG;
  const bool fp8 = c->weight_dtype == DFLASH_DTYPE_FP8_E4M3 || c->weight_dtype == DFLASH_DTYPE_FP4_E2M1;
  if (bad_ptr(w->tok_embd) || bad_ptr(w->lm_head) || bad_ptr(w->fc) || bad_ptr(w->hidden_norm) ||
      bad_ptr(w->out_norm))
    return DFLASH_ERR_INVALID_ARG;
  if (fp8 && !w->lm_head_scale) return DFLASH_ERR_INVALID_ARG;
  for (int l = 0; l < c->n_layer; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    const void* ps[] = {L.attn_norm, L.wq, L.wk, L.wv, L.wo, L.q_norm, L.k_norm, L.ffn_norm,
                        L.gate, L.up, L.down};
    for (const void* q : ps)
      if (bad_ptr(q)) return DFLASH_ERR_INVALID_ARG;
    if (fp8) {
      const float* sc[] = {L.wq_scale, L.wk_scale, L.wv_scale, L.wo_scale,
                           L.gate_scale, L.up_scale, L.down_scale};
      for (const float* q : sc)
        if (!q) return DFLASH_ERR_INVALID_ARG;
    }
  }
  return DFLASH_OK;
}

}  // namespace

extern "C" {

int dflash_workspace_size(const dflash_config* cfg, size_t* ring_bytes, size_t* scratch_bytes) {
  const int v = validate(cfg);
  if (v != DFLASH_OK) return v;
  if (!ring_bytes || !scratch_bytes) return DFLASH_ERR_INVALID_ARG;
  const Layout L = layout(*cfg);
  *ring_bytes = L.ring_total;
  *scratch_bytes = L.total;
  return DFLASH_OK;
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, void* ring_mem,
                  void* scratch_mem, dflash_handle** out) {
  if (!out) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  int v = validate(cfg);
  if (v != DFLASH_OK) return v;
  if ((v = check_weights(cfg, w)) != DFLASH_OK) return v;
  if (!ring_mem || !scratch_mem || (reinterpret_cast<uintptr_t>(ring_mem) & (kAlign - 1)) ||
      (reinterpret_cast<uintptr_t>(scratch_mem) & (kAlign - 1)))
    return DFLASH_ERR_INVALID_ARG;
  clear_stale_error();
  dflash_handle* h = new (std::nothrow) dflash_handle();
  if (!h) return DFLASH_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->w = *w;
  h->g = geometry(*cfg);
  h->L = layout(*cfg);
  h->ring = static_cast<char*>(ring_mem);
  h->scratch = static_cast<char*>(scratch_mem);
  h->err[0] = 0;
  // host fp64 inverse-frequency table theta^(-2j/head_dim)
  const int half = cfg->head_dim / 2;
  double inv[64];
  for (int j = 0; j < half; ++j) inv[j] = std::pow(cfg->rope_theta, -2.0 * j / cfg->head_dim);
  cudaError_t e = cudaMemcpy(h->S<double>(h->L.inv_freq), inv, sizeof(double) * half,
                             cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(h->scratch + h->L.counters, 0, sizeof(int) * h->L.n_counters);
  if (e == cudaSuccess) e = cudaMemset(h->scratch + h->L.attn_cnt, 0, sizeof(int) * 2 * h->L.attn_groups);
  // chain tickets, flags and counters (contiguous: tickets, flags, counts, done)
  if (e == cudaSuccess)
    e = cudaMemset(h->scratch + h->L.chain_cnt, 0, h->L.chain_done + sizeof(int) - h->L.chain_cnt);
  if (e == cudaSuccess) e = cudaMemset(h->scratch + h->L.status, 0, sizeof(unsigned));
  // zero K/V (empty slots are masked, but p = 0 times a NaN left in reused memory
  // is NaN) and mark every slot empty
  if (e == cudaSuccess) e = cudaMemset(h->ring, 0, h->L.ring_kv_bytes * cfg->max_seq);
  if (e == cudaSuccess)
    e = launch_fill_i32(h->ring_pos(0), cfg->max_seq * cfg->window, -1, nullptr);
  if (e == cudaSuccess) e = configure_gemm(kXkMax);
  if (e == cudaSuccess) e = configure_gemm_tma();
  if (e == cudaSuccess) e = configure_gemm_fp4();
  if (e == cudaSuccess) e = configure_gemm_umma();
  if (e == cudaSuccess && !build_maps(h)) e = cudaErrorNotSupported;
  if (e == cudaSuccess)
    e = configure_attention(cfg->n_head / cfg->n_head_kv, cfg->head_dim,
                            cfg->ring_dtype == DFLASH_DTYPE_F32, cfg->window, cfg->n_head_kv);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking);
  // the chain's waits need its whole grid resident at once
  // (chains run on the 16-row TMA kernel: not for FP4 and E4M3 weights, whose
  // projections run on the tensor-memory pipeline)
  if (e == cudaSuccess && h->g.wt != W_FP4 && h->g.wt != W_FP8)
    h->chain_ok = gemm_chain_capacity(h->g.wt) >= kGemmGrid;
  h->chain = false;   // opt-in: measured no faster than one launch per projection
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cuda_fail(h, e, "dflash_create");
    std::fprintf(stderr, "dflash_create: %s\n", h->err);
    if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
    delete h;
    return DFLASH_ERR_CUDA;
  }
  *out = h;
  return DFLASH_OK;
}

void dflash_destroy(dflash_handle* h) {
  if (!h) return;
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  for (int w = 0; w <= DFLASH_BLOCK; ++w) {
    if (h->execs[w]) cudaGraphExecDestroy(h->execs[w]);
    if (h->graphs[w]) cudaGraphDestroy(h->graphs[w]);
    if (h->loop_execs[w]) cudaGraphExecDestroy(h->loop_execs[w]);
    if (h->loop_graphs[w]) cudaGraphDestroy(h->loop_graphs[w]);
  }
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  delete h;
}

namespace {

// encode T rows (validated by the caller)
int run_encode(dflash_handle* h, const void* feats, int T, float* H_t, cudaStream_t st) {
  const Geometry& g = h->g;
  GemmShape sh[2];
  inject_shapes(g, sh);
  const int n_mb = cdiv(T, 16);
  GemmParams p = base_params(h);
  CUtensorMap fm;
  if (h->enc_dense && T >= 128 && make_map(&fm, feats, W_BF16, g.fdim, T, 64, 128, true)) {
    // >= 128 rows: a dense contraction on the tcgen05 kernel (bf16 features
    // are exact in bf16: no lo part)
    p.tm_xh = fm;
    p.tm_xl = fm;
    p.has_lo = 0;
    p.tm_w[0] = h->td_fc;
    p.seg[0] = {h->w.fc, nullptr, 0, g.d};
    p.nseg = 1; p.N = g.d; p.map = MAP_SEGMENTS; p.M = T; p.K = g.fdim;
    p.n_tiles = cdiv(g.d, kTileRows); p.n_mb = n_mb; p.cpt = cdiv(g.fdim, 64);
    p.epi = EPI_STORE_SS; p.out = h->S<float>(h->L.inj_raw); p.ldo = g.d;
    p.ss_out = h->S<float>(h->L.inj_ss); p.ss_out_ld = h->L.ss_ld;
    prof_begin(h, PC_ENCODE, st);
    DF_CHECK(h, launch_gemm_umma(W_BF16, p, st));
    DF_CHECK(h, launch_rms_apply(h->S<float>(h->L.inj_raw), h->S<float>(h->L.inj_ss), p.n_tiles,
                                 h->L.ss_ld, T, g.d, h->w.hidden_norm, g.dense_bf16, h->cfg.eps, H_t,
                                 st));
    prof_end(h, st);
    return DFLASH_OK;
  }
  set_plan(p, sh[0], n_mb);
  p.x = feats; p.x_mode = g.dense_bf16 ? X_BF16 : X_F32; p.ldx = g.fdim; p.M = T;
  p.seg[0] = {h->w.fc, nullptr, 0, g.d};
  p.nseg = 1; p.N = g.d; p.map = MAP_SEGMENTS;
  p.epi = EPI_STORE_SS; p.out = h->S<float>(h->L.inj_raw); p.ldo = g.d;
  p.ss_out = h->S<float>(h->L.inj_ss); p.ss_out_ld = h->L.ss_ld;
  prof_begin(h, PC_ENCODE, st);
  DF_CHECK(h, launch_gemm(g.dense_bf16 ? W_BF16 : W_F32, p, st));
  DF_CHECK(h, launch_rms_apply(h->S<float>(h->L.inj_raw), h->S<float>(h->L.inj_ss), sh[0].n_tiles,
                               h->L.ss_ld, T, g.d, h->w.hidden_norm, g.dense_bf16, h->cfg.eps, H_t,
                               st));
  prof_end(h, st);
  return DFLASH_OK;
}

// inject T rows: into sequence `seq`'s ring, or (rows_per_seq > 0) row t into
// sequence t / rows_per_seq, only its first count[sequence] rows
int run_inject(dflash_handle* h, int seq, const float* H_t, const int32_t* pos, int T,
               int rows_per_seq, const int32_t* count, cudaStream_t st) {
  const Geometry& g = h->g;
  GemmShape sh[2];
  inject_shapes(g, sh);
  float2* rope = h->S<float2>(h->L.inj_rope);
  prof_begin(h, PC_INJECT, st);
  DF_CHECK(h, launch_rope_table(pos, T, h->S<double>(h->L.inv_freq), g.hd, rope, h->ring_pos(seq),
                                g.W, rows_per_seq, count, h->status(), st));
  const int n_mb = cdiv(T, 16);
  GemmParams p = base_params(h);
  if (g.wt == W_FP4) {
    // FP4 weights: H_t as an fp16 pair, then per layer its wk / wv projection on
    // the 16-row TMA kernel with the ring scatter in the epilogue (the ring
    // pointer moved to the layer's planes: the epilogue's layer 0)
    DF_CHECK(h, launch_split_pair(H_t, T * g.d, h->S<uint16_t>(h->L.inj_hi),
                                  h->S<uint16_t>(h->L.inj_lo), pair_f16_of(g, T), st));
    const size_t layer_bytes = h->L.ring_kv_bytes / g.L;
    const GemmShape kv = {cdiv(2 * g.kvd, kTileRows), g.d, tma_chunk_k(g.wt)};
    for (int l = 0; l < g.L; ++l) {
      const dflash_layer_weights& lw = h->w.layers[l];
      GemmParams q = base_params(h);
      set_plan(q, kv, n_mb);
      q.tm_xh = h->tm_inj[0];
      q.tm_xl = h->tm_inj[1];
      q.has_lo = 1;
      q.tm_w[0] = h->tm_layer[l][1];
      q.tm_w[1] = h->tm_layer[l][2];
      q.tm_w64[0] = h->tm_layer64[l][1];
      q.tm_w64[1] = h->tm_layer64[l][2];
      q.tm_s64[0] = h->tm_scale64[l][1];
      q.tm_s64[1] = h->tm_scale64[l][2];
      q.w64 = 1;
      if (h->x4) {
        q.tm_x4 = h->tm_x4[3];
        q.x4 = 1;
      }
      q.seg[0] = {lw.wk, lw.wk_scale, 0, g.kvd};
      q.seg[1] = {lw.wv, lw.wv_scale, g.kvd, g.kvd};
      q.k_norm_l[0] = lw.k_norm;
      q.nseg = 2; q.N = 2 * g.kvd; q.map = MAP_SEGMENTS; q.M = T;
      q.epi = EPI_INJECT; q.ring_seq = h->ring_seq(seq) + (size_t)l * layer_bytes; q.pos = pos;
      q.rope_cs = rope;
      q.rows_per_seq = rows_per_seq; q.row_count = count; q.ring_seq_stride = h->L.ring_seq_bytes;
      DF_CHECK(h, launch_gemm_fp4(W_FP4, q, st));
    }
    prof_end(h, st);
    return DFLASH_OK;
  }
  if (h->inj_dense && T >= 128) {
    // >= 128 rows: H_t as a 16-bit hi/lo pair, then per layer its wk / wv
    // projection on the tcgen05 kernel with the ring scatter in the epilogue
    // (the ring pointer moved to the layer's planes: the epilogue's layer 0)
    DF_CHECK(h, launch_split_pair(H_t, T * g.d, h->S<uint16_t>(h->L.inj_hi),
                                  h->S<uint16_t>(h->L.inj_lo), pair_f16_of(g, T), st));
    const size_t layer_bytes = h->L.ring_kv_bytes / g.L;
    for (int l = 0; l < g.L; ++l) {
      const dflash_layer_weights& lw = h->w.layers[l];
      GemmParams q = base_params(h);
      q.tm_xh = h->td_inj[0];
      q.tm_xl = h->td_inj[1];
      q.has_lo = 1;
      q.tm_w[0] = h->td_kv[l][0];
      q.tm_w[1] = h->td_kv[l][1];
      q.seg[0] = {lw.wk, lw.wk_scale, 0, g.kvd};
      q.seg[1] = {lw.wv, lw.wv_scale, g.kvd, g.kvd};
      q.k_norm_l[0] = lw.k_norm;
      q.nseg = 2; q.N = 2 * g.kvd; q.map = MAP_SEGMENTS; q.M = T; q.K = g.d;
      q.n_tiles = cdiv(2 * g.kvd, kTileRows); q.n_mb = n_mb; q.cpt = cdiv(g.d, 64);
      q.epi = EPI_INJECT; q.ring_seq = h->ring_seq(seq) + (size_t)l * layer_bytes; q.pos = pos;
      q.rope_cs = rope;
      q.rows_per_seq = rows_per_seq; q.row_count = count; q.ring_seq_stride = h->L.ring_seq_bytes;
      DF_CHECK(h, launch_gemm_umma(g.wt, q, st));
    }
    prof_end(h, st);
    return DFLASH_OK;
  }
  set_plan(p, sh[1], n_mb);
  p.x = H_t; p.x_mode = X_F32; p.ldx = g.d; p.M = T;
  for (int l = 0; l < g.L; ++l) {
    const dflash_layer_weights& lw = h->w.layers[l];
    p.seg[2 * l] = {lw.wk, lw.wk_scale, 2 * l * g.kvd, g.kvd};
    p.seg[2 * l + 1] = {lw.wv, lw.wv_scale, 2 * l * g.kvd + g.kvd, g.kvd};
    p.k_norm_l[l] = lw.k_norm;
  }
  p.nseg = 2 * g.L; p.N = 2 * g.L * g.kvd; p.map = MAP_SEGMENTS;
  p.epi = EPI_INJECT; p.ring_seq = h->ring_seq(seq); p.pos = pos; p.rope_cs = rope;
  p.rows_per_seq = rows_per_seq; p.row_count = count; p.ring_seq_stride = h->L.ring_seq_bytes;
  DF_CHECK(h, launch_gemm(g.wt, p, st));
  prof_end(h, st);
  return DFLASH_OK;
}

// accept + bonus token + position update, then encode and inject the accepted
// rows of every sequence (validated by the caller)
int run_advance(dflash_handle* h, int n_seq, const int32_t* drafts, const int32_t* targets,
                const void* feats, int32_t* id_last, int32_t* n_past, int32_t* n_ok,
                cudaStream_t st) {
  int32_t* pos = h->S<int32_t>(h->L.loop_pos);
  int32_t* cnt = h->S<int32_t>(h->L.loop_cnt);
  float* H = h->S<float>(h->L.loop_H);
  const int T = n_seq * DFLASH_BLOCK;
  PROF(h, PC_ACCEPT, st, launch_advance(drafts, targets, n_seq, h->width, id_last, n_past, n_ok, pos, cnt, st));
  int rc = run_encode(h, feats, T, H, st);
  if (rc != DFLASH_OK) return rc;
  return run_inject(h, 0, H, pos, T, DFLASH_BLOCK, cnt, st);
}

int check_advance(const dflash_handle* h, int n_seq) {
  if (n_seq < 1 || n_seq > h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  if (n_seq * DFLASH_BLOCK > h->g.max_inject || h->g.W < DFLASH_BLOCK) return DFLASH_ERR_TOO_MANY_ROWS;
  return DFLASH_OK;
}

}  // namespace

int dflash_encode(dflash_handle* h, const void* feats, int32_t T, float* H_t, void* stream) {
  clear_stale_error();
  if (!h || T < 0) return DFLASH_ERR_INVALID_ARG;
  if (T > h->g.max_inject) return DFLASH_ERR_TOO_MANY_ROWS;
  if (T == 0) return DFLASH_OK;
  if (bad_ptr(feats) || bad_ptr(H_t)) return DFLASH_ERR_INVALID_ARG;
  return run_encode(h, feats, T, H_t, static_cast<cudaStream_t>(stream));
}

int dflash_inject(dflash_handle* h, int32_t seq, const float* H_t, const int32_t* pos, int32_t T,
                  void* stream) {
  clear_stale_error();
  if (!h || T < 0) return DFLASH_ERR_INVALID_ARG;
  if (seq < 0 || seq >= h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  if (T > h->g.W || T > h->g.max_inject) return DFLASH_ERR_TOO_MANY_ROWS;
  if (T == 0) return DFLASH_OK;
  if (bad_ptr(H_t) || !pos) return DFLASH_ERR_INVALID_ARG;
  return run_inject(h, seq, H_t, pos, T, 0, nullptr, static_cast<cudaStream_t>(stream));
}

int dflash_advance(dflash_handle* h, int32_t n_seq, const int32_t* drafts, const int32_t* targets,
                   const void* feats, int32_t* id_last, int32_t* n_past, int32_t* n_ok,
                   void* stream) {
  clear_stale_error();
  if (!h) return DFLASH_ERR_INVALID_ARG;
  const int v = check_advance(h, n_seq);
  if (v != DFLASH_OK) return v;
  if (!drafts || !targets || bad_ptr(feats) || !id_last || !n_past || !n_ok)
    return DFLASH_ERR_INVALID_ARG;
  return run_advance(h, n_seq, drafts, targets, feats, id_last, n_past, n_ok,
                     static_cast<cudaStream_t>(stream));
}

int dflash_set_chain(dflash_handle* h, int32_t enable) {
  if (!h || h->capturing) return DFLASH_ERR_INVALID_ARG;
  if (enable && !h->chain_ok) return DFLASH_ERR_UNSUPPORTED;
  h->chain = enable != 0;
  return DFLASH_OK;
}

int dflash_attention_kernel(const dflash_handle* h, int32_t n_seq) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  const Geometry& g = h->g;
  AttnParams a;
  std::memset(&a, 0, sizeof(a));
  a.ring_bf16 = g.ring_bf16;
  a.n_head = g.Hq; a.n_head_kv = g.Hkv; a.hd = g.hd; a.window = g.W;
  a.part_o = h->S<float>(h->L.attn_part);
  a.plan_nv = h->S<int>(h->L.plan_nv);
  return attention_kind(a, n_seq);
}

int dflash_set_block_width(dflash_handle* h, int32_t width) {
  if (!h || width < 2 || width > DFLASH_BLOCK) return DFLASH_ERR_INVALID_ARG;
  if (h->capturing) return DFLASH_ERR_INVALID_ARG;
  h->width = width;
  return DFLASH_OK;
}

int dflash_step(dflash_handle* h, int32_t n_seq, const int32_t* id_last, const int32_t* n_past,
                float* logits, int32_t* drafts, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  if (!id_last || !n_past || !drafts) return DFLASH_ERR_INVALID_ARG;
  return run_step(h, n_seq, id_last, n_past, logits, drafts, static_cast<cudaStream_t>(stream));
}

int dflash_accept(dflash_handle* h, int32_t n_seq, const int32_t* drafts, const int32_t* targets,
                  int32_t* n_ok, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  if (!drafts || !targets || !n_ok) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  clear_stale_error();
  PROF(h, PC_ACCEPT, st, launch_accept(drafts, targets, n_ok, n_seq, h->width, nullptr, st));
  return DFLASH_OK;
}

int dflash_capture(dflash_handle* h, int32_t n_seq, const int32_t* id_last, const int32_t* n_past,
                   float* logits, int32_t* drafts, const int32_t* targets, int32_t* n_ok,
                   void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  if (!id_last || !n_past || !drafts || (!targets != !n_ok)) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // order the capture after the caller's queued work (nothing is launched here)
  DF_CHECK(h, cudaStreamSynchronize(st));
  {
    const int w = h->width;
    if (h->execs[w]) { cudaGraphExecDestroy(h->execs[w]); h->execs[w] = nullptr; }
    if (h->graphs[w]) { cudaGraphDestroy(h->graphs[w]); h->graphs[w] = nullptr; }
  }
  DF_CHECK(h, cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  h->capturing = true;
  int rc = run_step(h, n_seq, id_last, n_past, logits, drafts, h->cap_stream);
  if (rc == DFLASH_OK && targets) {
    cudaError_t e = launch_accept(drafts, targets, n_ok, n_seq, h->width,
                                  stamp_slot(h, PC_ACCEPT), h->cap_stream);
    if (e != cudaSuccess) rc = cuda_fail(h, e, "accept (capture)");
  }
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(h->cap_stream, &graph);
  h->capturing = false;
  if (rc != DFLASH_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamEndCapture");
  h->graphs[h->width] = graph;
  DF_CHECK(h, cudaGraphInstantiate(&h->execs[h->width], graph, 0));
  return DFLASH_OK;
}

int dflash_replay(dflash_handle* h, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (!h->execs[h->width]) return DFLASH_ERR_NOT_CAPTURED;
  DF_CHECK(h, cudaGraphLaunch(h->execs[h->width], static_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

int dflash_capture_loop(dflash_handle* h, int32_t n_seq, const int32_t* targets, const void* feats,
                        int32_t* id_last, int32_t* n_past, int32_t* n_ok, float* logits,
                        int32_t* drafts, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  const int v = check_advance(h, n_seq);
  if (v != DFLASH_OK) return v;
  if (!targets || bad_ptr(feats) || !id_last || !n_past || !n_ok || !drafts)
    return DFLASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DF_CHECK(h, cudaStreamSynchronize(st));
  {
    const int w = h->width;
    if (h->loop_execs[w]) { cudaGraphExecDestroy(h->loop_execs[w]); h->loop_execs[w] = nullptr; }
    if (h->loop_graphs[w]) { cudaGraphDestroy(h->loop_graphs[w]); h->loop_graphs[w] = nullptr; }
  }
  DF_CHECK(h, cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  h->capturing = true;
  int rc = run_advance(h, n_seq, drafts, targets, feats, id_last, n_past, n_ok, h->cap_stream);
  if (rc == DFLASH_OK) rc = run_step(h, n_seq, id_last, n_past, logits, drafts, h->cap_stream);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(h->cap_stream, &graph);
  h->capturing = false;
  if (rc != DFLASH_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamEndCapture");
  h->loop_graphs[h->width] = graph;
  DF_CHECK(h, cudaGraphInstantiate(&h->loop_execs[h->width], graph, 0));
  return DFLASH_OK;
}

int dflash_replay_loop(dflash_handle* h, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (!h->loop_execs[h->width]) return DFLASH_ERR_NOT_CAPTURED;
  DF_CHECK(h, cudaGraphLaunch(h->loop_execs[h->width], static_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

int dflash_graph_nodes(dflash_handle* h, int32_t loop, int32_t* kernels, int32_t* mem_alloc,
                       int32_t* other) {
  if (!h || !kernels || !mem_alloc || !other) return DFLASH_ERR_INVALID_ARG;
  cudaGraph_t g = loop ? h->loop_graphs[h->width] : h->graphs[h->width];
  if (!g) return DFLASH_ERR_NOT_CAPTURED;
  size_t n = 0;
  DF_CHECK(h, cudaGraphGetNodes(g, nullptr, &n));
  std::vector<cudaGraphNode_t> nodes(n);
  if (n) DF_CHECK(h, cudaGraphGetNodes(g, nodes.data(), &n));
  int k = 0, m = 0, o = 0;
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType t;
    DF_CHECK(h, cudaGraphNodeGetType(nodes[i], &t));
    if (t == cudaGraphNodeTypeKernel) ++k;
    else if (t == cudaGraphNodeTypeMemAlloc || t == cudaGraphNodeTypeMemFree) ++m;
    else ++o;
  }
  *kernels = k;
  *mem_alloc = m;
  *other = o;
  return DFLASH_OK;
}

int dflash_step_host(dflash_handle* h, int32_t n_seq, const int32_t* id_last,
                     const int32_t* n_past, float* logits, int32_t* drafts, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  if (!id_last || !n_past || !drafts) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* d_idl = h->S<int32_t>(h->L.idl_int);
  int32_t* d_np = h->S<int32_t>(h->L.npast_int);
  int32_t* d_dr = h->S<int32_t>(h->L.drafts_int);
  float* d_lg = logits ? h->S<float>(h->L.logits_int) : nullptr;
  DF_CHECK(h, cudaMemcpyAsync(d_idl, id_last, sizeof(int32_t) * n_seq, cudaMemcpyHostToDevice, st));
  DF_CHECK(h, cudaMemcpyAsync(d_np, n_past, sizeof(int32_t) * n_seq, cudaMemcpyHostToDevice, st));
  const int rc = run_step(h, n_seq, d_idl, d_np, d_lg, d_dr, st);
  if (rc != DFLASH_OK) return rc;
  DF_CHECK(h, cudaMemcpyAsync(drafts, d_dr, sizeof(int32_t) * n_seq * (DFLASH_BLOCK - 1),
                              cudaMemcpyDeviceToHost, st));
  if (logits)
    DF_CHECK(h, cudaMemcpyAsync(logits, d_lg, sizeof(float) * (size_t)n_seq * DFLASH_BLOCK * h->g.V,
                                cudaMemcpyDeviceToHost, st));
  DF_CHECK(h, cudaStreamSynchronize(st));
  return DFLASH_OK;
}

int dflash_ring_reset(dflash_handle* h, int32_t seq, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (seq < 0 || seq >= h->g.max_seq) return DFLASH_ERR_SEQ_RANGE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DF_CHECK(h, cudaMemsetAsync(h->ring_seq(seq), 0, h->L.ring_seq_bytes, st));
  DF_CHECK(h, launch_fill_i32(h->ring_pos(seq), h->g.W, -1, st));
  return DFLASH_OK;
}

int dflash_read_status(dflash_handle* h, uint32_t* status, void* stream) {
  if (!h || !status) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  DF_CHECK(h, cudaStreamSynchronize(st));
  DF_CHECK(h, cudaMemcpy(&v, h->status(), sizeof(unsigned), cudaMemcpyDeviceToHost));
  DF_CHECK(h, cudaMemset(h->status(), 0, sizeof(unsigned)));
  *status = v;
  return v ? DFLASH_ERR_DEVICE : DFLASH_OK;
}

int dflash_profile_enable(dflash_handle* h, int enable) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (h->capturing || enable < 0 || enable > 2) return DFLASH_ERR_INVALID_ARG;
  h->prof = enable == 1;
  h->stamps = enable == 2;
  return DFLASH_OK;
}

int dflash_profile_stamps(dflash_handle* h, int32_t max, int32_t* cls, double* start_us,
                          double* end_us, int32_t* n, void* stream) {
  if (!h || !cls || !start_us || !end_us || !n || max < 0) return DFLASH_ERR_INVALID_ARG;
  const int k = std::min<int>(max, (int)h->stamp_cls.size());
  std::vector<unsigned long long> raw(2 * (size_t)std::max(k, 1));
  DF_CHECK(h, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  if (k) DF_CHECK(h, cudaMemcpy(raw.data(), h->scratch + h->L.stamps, sizeof(unsigned long long) * 2 * k,
                                cudaMemcpyDeviceToHost));
  unsigned long long t0 = ~0ull;
  for (int i = 0; i < k; ++i)
    if (raw[2 * i + 1]) t0 = std::min(t0, ~raw[2 * i]);
  for (int i = 0; i < k; ++i) {
    cls[i] = h->stamp_cls[i];
    const bool ran = raw[2 * i + 1] != 0;
    start_us[i] = ran ? (double)(~raw[2 * i] - t0) * 1e-3 : -1.0;
    end_us[i] = ran ? (double)(raw[2 * i + 1] - t0) * 1e-3 : -1.0;
  }
  *n = k;
  return DFLASH_OK;
}

int dflash_profile_read(dflash_handle* h, double* ms, int32_t* launches) {
  if (!h || !ms || !launches) return DFLASH_ERR_INVALID_ARG;
  for (int i = 0; i < DFLASH_PROF_N; ++i) {
    ms[i] = 0.0;
    launches[i] = 0;
  }
  for (const auto& r : h->recs) {
    DF_CHECK(h, cudaEventSynchronize(r.b));
    float t = 0.f;
    DF_CHECK(h, cudaEventElapsedTime(&t, r.a, r.b));
    ms[r.cls] += t;
    launches[r.cls] += (r.cls == PC_ENCODE) ? 2 : (r.cls == PC_INJECT ? 2 : 1);
  }
  h->recs.clear();
  h->ev_used = 0;
  return DFLASH_OK;
}

const char* dflash_status_string(int s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED: return "unsupported geometry or dtype";
    case DFLASH_ERR_TOO_MANY_ROWS: return "too many rows (T > window or T > max_inject)";
    case DFLASH_ERR_SEQ_RANGE: return "sequence index out of range";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_NOT_CAPTURED: return "no captured graph";
    case DFLASH_ERR_DEVICE: return "device status flag set";
  }
  return "unknown status";
}

const char* dflash_last_error(const dflash_handle* h) { return h ? h->err : ""; }

}  // extern "C"
