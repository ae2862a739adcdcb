// Internal interface between the C-ABI layer and the kernels of libdflash.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dflash {

// weight storage of a projection matrix
enum WType { W_F32 = 0, W_BF16 = 1, W_FP8 = 2, W_FP4 = 3 };
// activation storage fed to a projection kernel
enum XMode { X_F32 = 0, X_BF16 = 1, X_F32_DENSE = 2 };
// what the split-K fix-up does with a finished 16 x 128 output tile
enum Epi {
  EPI_STORE = 0,     // out[m][n] = y
  EPI_STORE_SS = 1,  // out[m][n] = y; ss_out[tile][m] = sum over the tile of y^2
  EPI_RESID_SS = 2,  // out[m][n] += y; ss_out[tile][m] = sum over the tile of out^2
  EPI_SWIGLU = 3,    // out[m][f] = silu(gate) * up (tile = 64 gate rows + 64 up rows)
  EPI_QKV = 4,       // per-head RMSNorm + rope of q/k, raw v, into the block buffers
  EPI_INJECT = 5,    // per-head RMSNorm + rope of k, raw v, scattered into the ring
  EPI_LOGITS = 6     // logits + argmax partials; the last tile emits the drafts
};
enum RowMap { MAP_SEGMENTS = 0, MAP_SWIGLU = 1 };

// Programmatic dependent launch between the step's kernels: a projection's
// CTAs start (mbarrier set-up, first weight stages in flight) while the
// previous kernel's last CTAs finish their fix-up and epilogue; everything
// that reads an earlier kernel's output waits at griddepcontrol.wait, which
// returns only once that kernel has completed and its writes are visible.
// Measured 1.042 vs 1.065 ms per real-dimension step in the replayed graph.
constexpr bool kDependentLaunch = true;

constexpr int kTileRows = 128;     // output rows (weight rows) of one CTA tile
constexpr int kGemmThreads = 256;  // 8 warps x 16 weight rows
constexpr int kMaxSeg = 2 * 16;
constexpr int kMaxLayers = 16;
// widest activation stage (k extent) of the register-fed projection kernel:
// configure_gemm raises its shared-memory limit to this width, and every caller
// (the handle-based calls and the allocation-free encode) plans within it
constexpr int kGemmXkMax = 960;

struct GemmSeg {
  const void* w;        // [rows][K] row-major, weight dtype
  const float* scale;   // FP8: per-row scale; else null
  int row0;             // first virtual output row of this segment
  int rows;
};

struct GemmParams {
  // TMA path: tensor maps of the weight segments and of the activation pair
  CUtensorMap tm_w[4];
  // the same weights in 64-row boxes (one copy for four 16-row groups; bf16 and
  // E4M3 16-row kernel), used when w64 is set
  CUtensorMap tm_w64[4];
  CUtensorMap tm_s64[4];    // FP4: the block scales of 64 rows x 256 k per box
  int w64;
  CUtensorMap tm_xh;
  CUtensorMap tm_xl;
  // FP4 kernel: the activation pair as one 4-D tensor [K/64][hi, lo][rows][64]
  // (boxes of 64 k x 16 rows x hi+lo x 4: a stage's 256 k in one copy); x4 set
  CUtensorMap tm_x4;
  int x4;
  int has_lo;
  // activations: x[m][k], m < M, row stride ldx (elements)
  const void* x;
  int x_mode;
  int ldx;
  int M;
  int K;
  // RMSNorm of the activation rows: inv_rms[m] = 1 / sqrt(sum_p ss[p * ss_ld + m]
  // / rms_len + eps).  Raw inputs apply x * inv_rms * normw while staging; pre-split
  // inputs (x = h * normw, made by the producer) apply inv_rms to the output rows
  // (row_scale).
  const float* ss;
  int n_ss;
  int ss_ld;
  int rms_len;
  const void* normw;
  int norm_bf16;
  float eps;
  int row_scale;
  // weights
  GemmSeg seg[kMaxSeg];
  int nseg;
  int N;      // virtual output rows
  int map;
  // stream-K schedule (see gemm.cu)
  int n_tiles;  // 128-row output tiles
  int n_mb;     // 16-row activation blocks
  int cpt;      // k chunks per tile
  int grid;     // CTAs (one resident wave)
  int xk;       // k extent of one shared-memory activation stage
  float* partial;  // [2 * grid][16][128]
  int* counters;   // [n_tiles * n_mb], zero between launches
  // epilogue
  int epi;
  float* out;
  int ldo;
  float* ss_out;
  int ss_out_ld;
  // bf16 hi/lo pair output for the next projection (EPI_RESID_SS: split(out * pair_norm);
  // EPI_SWIGLU: split(silu(g) u)), row stride pair_ld
  uint16_t* pair_hi;
  uint16_t* pair_lo;
  int pair_ld;
  int pair_f16;           // the pair is fp16 (FP4 or E4M3 weights), else bf16
  const void* pair_norm;
  // q/k/v epilogues
  float* kblk;
  float* vblk;
  int qd, kvd, hd;
  const void* q_norm;
  const void* k_norm;
  const float2* rope_cs;  // [row][hd/2] (cos, sin)
  // injection epilogue
  void* ring_seq;         // this sequence's ring: [L][2][Hkv][W][hd]
  int ring_bf16;
  int window;
  int n_head_kv;
  const int32_t* pos;     // [T]
  // batched injection: row t belongs to sequence t / rows_per_seq (ring at
  // ring_seq + sequence x ring_seq_stride bytes); rows at or past
  // row_count[sequence] within their sequence are not written
  int rows_per_seq;
  const int32_t* row_count;
  unsigned long long ring_seq_stride;
  const void* k_norm_l[kMaxLayers];
  unsigned* status;
  // logits epilogue
  float2* am_part;        // [n_tiles][M] (value, index bits)
  int* am_counter;        // [M/16] finished tiles of each 16-row block, zero between launches
  int32_t* drafts;        // [M/16][15]; rows at or past block_width draft -1
  int block_width;
  // L2 prefetch of the next kernel's input (pf_count ranges of pf_bytes at
  // pf_stride), shared out over the CTAs once their weight stream is issued
  const char* pf_base;
  unsigned long long pf_bytes, pf_stride;
  int pf_count;
  unsigned long long* stamp;  // launch timestamp slot (profiling captures), else null
};

struct AttnParams {
  // bf16 ring with hd >= 64: the whole ring as a 2-D bf16 tensor [rows][hd]
  // (row = ((((seq L + layer) 2 + k|v) Hkv + kv head) W + slot), 64 x 64 boxes,
  // 128-byte swizzle; the kernel stages 64-slot sub-chunks with it
  CUtensorMap tm_ring;
  const float* q;         // [M][qd], roped
  const float* kblk;      // [M][kvd], roped
  const float* vblk;      // [M][kvd]
  const void* ring;       // all rings: [max_seq][L][2][Hkv][W][hd]
  const int32_t* ring_pos;  // [max_seq][W]
  const int32_t* n_past;  // [n_seq]
  int ring_bf16;
  int layer, n_layer;
  int n_head, n_head_kv, hd, window;
  float scale;
  int hpc;                // query heads per CTA (set by the launcher)
  int kq;                 // key lanes: warps per head
  int nb;                 // 64-key sub-chunk staging buffers (a multiple of kq)
  uint16_t* out_hi;       // [M][qd] hi/lo pair (the o projection's input)
  uint16_t* out_lo;
  int pair_f16;           // fp16 pair (FP4 or E4M3 weights), else bf16
  unsigned* status;       // device status bits (DFLASH_DEV_TIMEOUT on a copy that never lands)
  int block_width;        // block rows that exist (2..16): block keys at or past it are masked
  unsigned long long* stamp;  // launch timestamp slot (profiling captures), else null
  // split-window kernel: partial rows [CTA][16 hpc][hd] (+ (max, sum) per row) of
  // at most kAttnSplitMaxCtas CTAs, and two counters per (sequence, kv head, head
  // group), zero between launches (null: the cluster kernel always)
  float* part_o;
  float2* part_ml;
  int* counters;
  int n_seq;              // sequences of the step (set by the launcher)
  // stream-K kernel: the step's plan (attn_plan_kernel): listed sub-chunks per
  // sequence [n_seq] and their indices [n_seq][64] (null: no stream-K)
  int* plan_nv;
  int* plan_sub;
  // L2 prefetch of the next projection's weights (one contiguous range, null:
  // none), shared out over the CTAs once the q/k/v kernel has completed: the
  // attention reads little from HBM, the o projection then streams from L2
  const char* pf_base;
  unsigned long long pf_bytes;
};

// attention kernel of a step: split window (one resident wave), stream-K over
// all groups' windows (larger batches), or clusters with a DSMEM merge
enum AttnKind { ATTN_SPLIT = 0, ATTN_CLUSTER = 1, ATTN_STREAM = 2 };
int attention_kind(const AttnParams& p, int n_seq);
// the step's stream-K plan (before the step's first projection, when
// attention_kind is ATTN_STREAM)
cudaError_t launch_attention_plan(const AttnParams& p, int n_seq, cudaStream_t st);
constexpr int kAttnStreamMaxSeq = 1024;   // sequences of a stream-K step (its shared plan table)

// split-window attention: largest grid (CTAs) it is launched with, and the
// largest rows x head_dim of one CTA's partial (16 rows x 4 heads x 128); the
// stream-K kernel keeps two partials per CTA in the same scratch
constexpr int kAttnSplitMaxCtas = 512;
constexpr int kAttnPartFloats = 64 * 128;

size_t gemm_smem_bytes(int wt, int xk);
cudaError_t configure_gemm(int xk_max);
cudaError_t launch_gemm(int wt, const GemmParams& p, cudaStream_t st);

// A chain of 16-row projections in one persistent launch of the TMA kernel:
// phase k + 1 reads the activation pair phase k's epilogues write.  Every CTA
// walks its stream-K range of phase 0, then of phase 1, ...; the copies of a
// phase's activation chunk wait (bounded) for the flags of the previous phase's
// items that produce it, and a phase whose epilogue applies the 1/rms row scale
// waits for all of the previous phase's items of its 16-row block (their sums
// of squares).  Weight copies never wait on activations.  Every phase has its
// own partial tiles and tickets; the grid is one resident wave (every wait ends).
constexpr int kChainMax = 4;
template <int NPH>
struct ChainParams {
  GemmParams ph[NPH];
  int n_phase;
  int* item_done;    // [NPH][item_stride]: 1 once the item's epilogue stores are visible
  int* all_done;     // [NPH][mb_stride]: finished items of each 16-row block
  int* chain_done;   // CTAs past the chain; the last one clears flags and counters
  int item_stride, mb_stride;
};

size_t gemm_tma_smem_bytes(int wt);
cudaError_t configure_gemm_tma();
cudaError_t launch_gemm_tma(int wt, const GemmParams& p, cudaStream_t st);
// CTAs of the chain kernel the GPU holds at once (occupancy x SMs)
int gemm_chain_capacity(int wt);
cudaError_t launch_gemm_chain(int wt, const ChainParams<kChainMax>& cp, cudaStream_t st);
int tma_chunk_k(int wt);   // k per pipeline stage of the TMA projection kernel

// FP4 projection on tcgen05 with the decoded weights in tensor memory (16-row
// activation blocks; the schedule fields as for the 16-row kernels, K % 256 == 0)
size_t gemm_fp4_smem_bytes();
cudaError_t configure_gemm_fp4();
cudaError_t launch_gemm_fp4(int wt, const GemmParams& p, cudaStream_t st);   // wt: W_FP4 or W_FP8

// tcgen05 projection for >= 128 activation rows (bf16 or E4M3 weights)
size_t gemm_umma_smem_bytes();
cudaError_t configure_gemm_umma();
cudaError_t launch_gemm_umma(int wt, const GemmParams& p, cudaStream_t st);


// one cluster per (sequence, kv head, query-head group), partials merged in
// distributed shared memory
int attn_cluster_size(int window);
// the largest dynamic shared memory any launch plan of this geometry uses
size_t attn_cluster_smem(int group, int hd, int ring_f32);
cudaError_t configure_attention_cluster(int group, int hd, int ring_f32, int window, int n_head_kv);
cudaError_t launch_attention_cluster(const AttnParams& p, int n_seq, cudaStream_t st);
// split-window kernel when the grid fits on the GPU at once (and p.part_o is
// set), else the cluster kernel
cudaError_t configure_attention(int group, int hd, int ring_f32, int window, int n_head_kv);
cudaError_t launch_attention(const AttnParams& p, int n_seq, cudaStream_t st);
// dynamic shared memory of the split-window kernel for this geometry
size_t attn_split_smem(int group, int hd, int ring_f32);

cudaError_t launch_embed(const void* tok_embd, int dense_bf16, int n_embd, int n_vocab,
                         int mask_token, const int32_t* id_last, const int32_t* n_past, int n_seq,
                         const double* inv_freq, int hd, float* h, float* ss, float2* rope_cs,
                         const void* norm0, uint16_t* x_hi, uint16_t* x_lo, int pair_f16,
                         int parts, int ss_ld, unsigned* status, unsigned long long* stamp,
                         cudaStream_t st);
cudaError_t launch_rope_table(const int32_t* pos, int T, const double* inv_freq, int hd,
                              float2* rope_cs, int32_t* ring_pos, int window, int rows_per_seq,
                              const int32_t* count, unsigned* status, cudaStream_t st);
cudaError_t launch_advance(const int32_t* drafts, const int32_t* targets, int n_seq, int width,
                           int32_t* id_last, int32_t* n_past, int32_t* n_ok, int32_t* pos,
                           int32_t* count, cudaStream_t st);
cudaError_t launch_rms_apply(const float* raw, const float* ss, int n_ss, int ss_ld, int T,
                             int n, const void* normw, int norm_bf16, float eps, float* out,
                             cudaStream_t st);
cudaError_t launch_accept(const int32_t* drafts, const int32_t* targets, int32_t* n_ok, int n_seq,
                          int width, unsigned long long* stamp, cudaStream_t st);
cudaError_t launch_fill_i32(int32_t* p, int n, int32_t v, cudaStream_t st);
// x (fp32, n values) -> bf16 hi + lo with x = hi + lo + O(2^-17 |x|) (pair_f16:
// fp16 hi + lo)
cudaError_t launch_split_pair(const float* x, int n, uint16_t* hi, uint16_t* lo, int pair_f16,
                              cudaStream_t st);

}  // namespace dflash
