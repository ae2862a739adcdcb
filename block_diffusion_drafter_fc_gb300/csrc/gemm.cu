// Weight-streaming projection kernel of the drafter step and of injection.
//
// y[m][n] = sum_k x[m][k] W[n][k] for a few rows m (16 per m-block) and many
// weight rows n: the dense projections q/k/v/o/gate/up/down and the LM head of
// the block step (dflash_head.rs, struct DflashLayer; dflash-ops model card,
// Method: fp32 arithmetic whatever the storage dtype), plus fc and the
// all-layer wk/wv of injection (dflash_head.rs field fused_kv_weight).
//
// Design:
//  * One CTA = 8 warps = a tile of 128 weight rows x one k-range; each warp owns
//    16 weight rows and streams them from HBM with 16-byte loads straight into
//    registers (two register stages in flight), so there is no shared-memory
//    round trip for the weights, which are ~99% of the step's bytes.
//  * The 16 activation rows of the k-range are staged once per CTA in shared
//    memory, RMS-normalised on the way in when the projection follows a norm,
//    and split into bf16 hi + lo parts (x = hi + lo + O(2^-17 |x|)).  Weights
//    in bf16 are exact in the tensor core, so W*hi + W*lo reproduces fp32 math;
//    fp32 weights are split the same way (three products), E4M3 weights are
//    widened to bf16 exactly and scaled per row in the epilogue.
//  * mma.sync m16n8k16 runs with the weights as the A operand (16 weight rows)
//    and the activations as B (8 rows per n-tile).  The k order inside a chunk
//    is permuted identically for A and B so that each lane's 16-byte load is one
//    contiguous piece of a weight row.
//  * Split-K across CTAs: each CTA writes its 16 x 128 partial tile; the last
//    CTA of a tile (atomic ticket) sums the partials in k order, so results are
//    deterministic and graph replays are bitwise identical, then runs the fused
//    epilogue (residual + sum of squares for the next RMSNorm, SwiGLU, per-head
//    q/k norm + rope, ring scatter, logits + argmax).
#include "common.cuh"
#include "internal.h"

#include <math_constants.h>

namespace dflash {

template <int WT>
struct WTraits;
template <>
struct WTraits<W_BF16> {
  static constexpr int EPL = 8, KC = 32, NV = 1, PAD = 32, ESZ = 2, U = 4;
};
template <>
struct WTraits<W_F32> {
  static constexpr int EPL = 8, KC = 32, NV = 2, PAD = 32, ESZ = 4, U = 2;
};
template <>
struct WTraits<W_FP8> {
  static constexpr int EPL = 16, KC = 64, NV = 1, PAD = 8, ESZ = 1, U = 4;
};

static int pad_of(int wt) { return wt == W_FP8 ? 8 : 32; }

size_t gemm_smem_bytes(int wt, int xk) {
  const size_t xs = (size_t)xk + pad_of(wt);
  return 2 * 16 * xs * sizeof(uint16_t) + 16 * kTileRows * sizeof(float) + 16 * sizeof(float) +
         kTileRows * sizeof(float);
}

// Weight row `local` of `tile` -> its first byte (null when the row is past N).
DF_DEVICE const uint8_t* map_row(const GemmParams& p, int tile, int local, int esz,
                                 const float** scale) {
  int s = 0, r = 0;
  if (p.map == MAP_SWIGLU) {
    s = local < kTileRows / 2 ? 0 : 1;
    r = tile * (kTileRows / 2) + (local & (kTileRows / 2 - 1));
    if (r >= p.seg[s].rows) return nullptr;
  } else {
    const int vr = tile * kTileRows + local;
    if (vr >= p.N) return nullptr;
    while (s + 1 < p.nseg && vr >= p.seg[s + 1].row0) ++s;
    r = vr - p.seg[s].row0;
  }
  *scale = p.seg[s].scale ? p.seg[s].scale + r : nullptr;
  return reinterpret_cast<const uint8_t*>(p.seg[s].w) + (size_t)r * p.K * esz;
}

// Activation rows m0..m0+15, columns [xs0, xs0+xlen) -> bf16 hi/lo in shared memory.
DF_DEVICE void stage_x(const GemmParams& p, uint16_t* xh, uint16_t* xl, int XS,
                       const float* inv_rms, int m0, int xs0, int xlen) {
  const int q4 = xlen >> 2;
  for (int idx = threadIdx.x; idx < 16 * q4; idx += blockDim.x) {
    const int m = idx / q4, c = (idx - m * q4) * 4;
    const int row = m0 + m, k = xs0 + c;
    uint2 hi = make_uint2(0, 0), lo = make_uint2(0, 0);
    if (row < p.M) {
      if (p.x_mode == X_BF16) {
        hi = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.x) +
                                             (size_t)row * p.ldx + k);
      } else {
        float4 f = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.x) +
                                                    (size_t)row * p.ldx + k);
        if (p.normw) {
          const float r = inv_rms[m];
          f.x = f.x * r * load_dense(p.normw, p.norm_bf16, k + 0);
          f.y = f.y * r * load_dense(p.normw, p.norm_bf16, k + 1);
          f.z = f.z * r * load_dense(p.normw, p.norm_bf16, k + 2);
          f.w = f.w * r * load_dense(p.normw, p.norm_bf16, k + 3);
        }
        split_bf16x2(f.x, f.y, hi.x, lo.x);
        split_bf16x2(f.z, f.w, hi.y, lo.y);
      }
    }
    *reinterpret_cast<uint2*>(xh + m * XS + c) = hi;
    *reinterpret_cast<uint2*>(xl + m * XS + c) = lo;
  }
}

// ------------------------------------------------------------------ chunk math

template <int WT>
struct Chunk;

template <>
struct Chunk<W_BF16> {
  // A: row g (16 B = 8 bf16), B: row g+8.  Two k16 steps.
  static DF_DEVICE void run(const uint4* A, const uint4* B, const uint16_t* xh, const uint16_t* xl,
                            int XS, int xoff, int g, bool has_lo, float (&acc)[2][4]) {
    const uint32_t a0[4] = {A[0].x, B[0].x, A[0].y, B[0].y};
    const uint32_t a1[4] = {A[0].z, B[0].z, A[0].w, B[0].w};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint4 h = *reinterpret_cast<const uint4*>(xh + (8 * j + g) * XS + xoff);
      mma_bf16_16816(acc[j], a0, h.x, h.y);
      mma_bf16_16816(acc[j], a1, h.z, h.w);
      if (has_lo) {
        const uint4 l = *reinterpret_cast<const uint4*>(xl + (8 * j + g) * XS + xoff);
        mma_bf16_16816(acc[j], a0, l.x, l.y);
        mma_bf16_16816(acc[j], a1, l.z, l.w);
      }
    }
  }
};

template <>
struct Chunk<W_F32> {
  // A[0..1]: row g (8 floats), B[0..1]: row g+8.  Weights split hi + lo too.
  static DF_DEVICE void run(const uint4* A, const uint4* B, const uint16_t* xh, const uint16_t* xl,
                            int XS, int xoff, int g, bool has_lo, float (&acc)[2][4]) {
    uint32_t ah[2][4], al[2][4];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const float4 fa = *reinterpret_cast<const float4*>(&A[s]);
      const float4 fb = *reinterpret_cast<const float4*>(&B[s]);
      split_bf16x2(fa.x, fa.y, ah[s][0], al[s][0]);
      split_bf16x2(fb.x, fb.y, ah[s][1], al[s][1]);
      split_bf16x2(fa.z, fa.w, ah[s][2], al[s][2]);
      split_bf16x2(fb.z, fb.w, ah[s][3], al[s][3]);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint4 h = *reinterpret_cast<const uint4*>(xh + (8 * j + g) * XS + xoff);
      const uint4 l = *reinterpret_cast<const uint4*>(xl + (8 * j + g) * XS + xoff);
      mma_bf16_16816(acc[j], ah[0], h.x, h.y);
      mma_bf16_16816(acc[j], ah[1], h.z, h.w);
      mma_bf16_16816(acc[j], al[0], h.x, h.y);
      mma_bf16_16816(acc[j], al[1], h.z, h.w);
      if (has_lo) {
        mma_bf16_16816(acc[j], ah[0], l.x, l.y);
        mma_bf16_16816(acc[j], ah[1], l.z, l.w);
      }
    }
  }
};

template <>
struct Chunk<W_FP8> {
  // A: row g (16 E4M3 codes), B: row g+8.  Four k16 steps.
  static DF_DEVICE void run(const uint4* A, const uint4* B, const uint16_t* xh, const uint16_t* xl,
                            int XS, int xoff, int g, bool has_lo, float (&acc)[2][4]) {
    const uint32_t* wa = reinterpret_cast<const uint32_t*>(&A[0]);
    const uint32_t* wb = reinterpret_cast<const uint32_t*>(&B[0]);
    uint32_t a[4][4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      a[s][0] = e4m3x2_to_bf16x2((uint16_t)(wa[s] & 0xffffu));
      a[s][1] = e4m3x2_to_bf16x2((uint16_t)(wb[s] & 0xffffu));
      a[s][2] = e4m3x2_to_bf16x2((uint16_t)(wa[s] >> 16));
      a[s][3] = e4m3x2_to_bf16x2((uint16_t)(wb[s] >> 16));
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint16_t* hrow = xh + (8 * j + g) * XS + xoff;
      const uint4 h0 = *reinterpret_cast<const uint4*>(hrow);
      const uint4 h1 = *reinterpret_cast<const uint4*>(hrow + 8);
      mma_bf16_16816(acc[j], a[0], h0.x, h0.y);
      mma_bf16_16816(acc[j], a[1], h0.z, h0.w);
      mma_bf16_16816(acc[j], a[2], h1.x, h1.y);
      mma_bf16_16816(acc[j], a[3], h1.z, h1.w);
      if (has_lo) {
        const uint16_t* lrow = xl + (8 * j + g) * XS + xoff;
        const uint4 l0 = *reinterpret_cast<const uint4*>(lrow);
        const uint4 l1 = *reinterpret_cast<const uint4*>(lrow + 8);
        mma_bf16_16816(acc[j], a[0], l0.x, l0.y);
        mma_bf16_16816(acc[j], a[1], l0.z, l0.w);
        mma_bf16_16816(acc[j], a[2], l1.x, l1.y);
        mma_bf16_16816(acc[j], a[3], l1.z, l1.w);
      }
    }
  }
};

template <int WT>
DF_DEVICE void load_stage(uint4 (&A)[WTraits<WT>::U][WTraits<WT>::NV], uint4 (&B)[WTraits<WT>::U][WTraits<WT>::NV],
                          const uint8_t* pa, const uint8_t* pb, int c0, int nch) {
  using T = WTraits<WT>;
#pragma unroll
  for (int u = 0; u < T::U; ++u) {
    const int c = c0 + u;
#pragma unroll
    for (int v = 0; v < T::NV; ++v) {
      const size_t off = (size_t)c * T::KC * T::ESZ + v * 16;
      A[u][v] = (pa && c < nch) ? ldg_stream(pa + off) : make_uint4(0, 0, 0, 0);
      B[u][v] = (pb && c < nch) ? ldg_stream(pb + off) : make_uint4(0, 0, 0, 0);
    }
  }
}

template <int WT>
DF_DEVICE void compute_stage(const uint4 (&A)[WTraits<WT>::U][WTraits<WT>::NV],
                             const uint4 (&B)[WTraits<WT>::U][WTraits<WT>::NV], const uint16_t* xh,
                             const uint16_t* xl, int XS, int c0, int nch, int g, int t, bool has_lo,
                             float (&acc)[2][4]) {
  using T = WTraits<WT>;
#pragma unroll
  for (int u = 0; u < T::U; ++u) {
    const int c = c0 + u;
    if (c < nch) Chunk<WT>::run(A[u], B[u], xh, xl, XS, c * T::KC + T::EPL * t, g, has_lo, acc);
  }
}

// ------------------------------------------------------------------ epilogues

DF_DEVICE void epilogue_rows(const GemmParams& p, float* acc_s, const float* scale_s, int mb,
                             int tile, int* s_flag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = mb * 16;
  const bool logits = p.epi == EPI_LOGITS;
  for (int i = tid; i < 16 * kTileRows; i += blockDim.x) {
    const int m = i / kTileRows, r = i - m * kTileRows;
    const int n = tile * kTileRows + r, row = m0 + m;
    float y = acc_s[i] * scale_s[r];
    if (n < p.N && row < p.M) {
      if (p.epi == EPI_RESID_SS) {
        float* o = p.out + (size_t)row * p.ldo + n;
        y += *o;
        *o = y;
      } else if (p.out) {
        p.out[(size_t)row * p.ldo + n] = y;
      }
    } else {
      y = logits ? -CUDART_INF_F : 0.f;
    }
    acc_s[i] = y;
  }
  __syncthreads();
  if (p.epi == EPI_STORE_SS || p.epi == EPI_RESID_SS) {
    for (int m = warp; m < 16; m += kGemmThreads / 32) {
      float s = 0.f;
      for (int r = lane; r < kTileRows; r += 32) s += acc_s[m * kTileRows + r] * acc_s[m * kTileRows + r];
      s = warp_sum(s);
      if (lane == 0 && m0 + m < p.M) p.ss_out[(size_t)tile * p.ss_out_ld + m0 + m] = s;
    }
  }
  if (!logits) return;
  for (int m = warp; m < 16; m += kGemmThreads / 32) {
    float v = -CUDART_INF_F;
    int idx = 0x7fffffff;
    for (int r = lane; r < kTileRows; r += 32) {
      const int n = tile * kTileRows + r;
      if (n < p.N) argmax_merge(v, idx, acc_s[m * kTileRows + r], n);
    }
    warp_argmax(v, idx);
    if (lane == 0 && m0 + m < p.M)
      p.am_part[(size_t)tile * p.M + m0 + m] = make_float2(v, __int_as_float(idx));
  }
  // the last finished tile of the whole launch reduces the argmax partials
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int total = p.n_tiles * p.n_mb;
    *s_flag = atomicAdd(p.am_counter, 1) == total - 1;
  }
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  for (int row = warp; row < p.M; row += kGemmThreads / 32) {
    const int i = row & 15;
    if (i == 0) continue;
    float v = -CUDART_INF_F;
    int idx = 0x7fffffff;
    for (int tt = lane; tt < p.n_tiles; tt += 32) {
      const float2 e = __ldcg(p.am_part + (size_t)tt * p.M + row);
      argmax_merge(v, idx, e.x, __float_as_int(e.y));
    }
    warp_argmax(v, idx);
    if (lane == 0) p.drafts[(row >> 4) * 15 + i - 1] = idx;
  }
  if (tid == 0) *p.am_counter = 0;
}

DF_DEVICE void epilogue_swiglu(const GemmParams& p, const float* acc_s, const float* scale_s,
                               int mb, int tile) {
  const int half = kTileRows / 2, F = p.seg[0].rows;
  for (int i = threadIdx.x; i < 16 * half; i += blockDim.x) {
    const int m = i / half, j = i - m * half;
    const int f = tile * half + j, row = mb * 16 + m;
    if (f >= F || row >= p.M) continue;
    const float gv = acc_s[m * kTileRows + j] * scale_s[j];
    const float uv = acc_s[m * kTileRows + half + j] * scale_s[half + j];
    p.out[(size_t)row * p.ldo + f] = gv / (1.f + expf(-gv)) * uv;
  }
}

// Per-head RMSNorm + NEOX rope of q/k (raw v) for the block (EPI_QKV) or for
// injected context rows scattered into the ring (EPI_INJECT).
DF_DEVICE void epilogue_heads(const GemmParams& p, const float* acc_s, const float* scale_s,
                              int mb, int tile) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hd = p.hd, half = hd >> 1, hpt = kTileRows / hd;
  for (int item = warp; item < 16 * hpt; item += kGemmThreads / 32) {
    const int m = item / hpt, hh = item - m * hpt;
    const int n0 = tile * kTileRows + hh * hd, row = mb * 16 + m;
    if (n0 >= p.N || row >= p.M) continue;
    int kind, layer = 0, head = 0;
    const void* normw;
    if (p.epi == EPI_QKV) {
      kind = n0 < p.qd ? 0 : (n0 < p.qd + p.kvd ? 1 : 2);
      normw = kind == 0 ? p.q_norm : p.k_norm;
    } else {
      layer = n0 / (2 * p.kvd);
      const int w = n0 - layer * 2 * p.kvd;
      kind = w < p.kvd ? 1 : 2;
      head = (w - (kind == 2 ? p.kvd : 0)) / hd;
      normw = p.k_norm_l[layer];
    }
    const float* src = acc_s + m * kTileRows + hh * hd;
    const float* sc = scale_s + hh * hd;
    float x1[4], x2[4];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = lane + 32 * u;
      x1[u] = j < half ? src[j] * sc[j] : 0.f;
      x2[u] = j < half ? src[j + half] * sc[j + half] : 0.f;
      ss += x1[u] * x1[u] + x2[u] * x2[u];
    }
    if (kind != 2) {
      ss = warp_sum(ss);
      const float inv = 1.f / sqrtf(ss / (float)hd + p.eps);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = lane + 32 * u;
        if (j >= half) continue;
        const float a = x1[u] * inv * load_dense(normw, p.norm_bf16, j);
        const float b = x2[u] * inv * load_dense(normw, p.norm_bf16, j + half);
        const float2 cs = p.rope_cs[(size_t)row * half + j];
        x1[u] = a * cs.x - b * cs.y;
        x2[u] = b * cs.x + a * cs.y;
      }
    }
    if (p.epi == EPI_QKV) {
      float* dst = kind == 0 ? p.out + (size_t)row * p.qd + n0
                 : kind == 1 ? p.kblk + (size_t)row * p.kvd + (n0 - p.qd)
                             : p.vblk + (size_t)row * p.kvd + (n0 - p.qd - p.kvd);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = lane + 32 * u;
        if (j < half) {
          dst[j] = x1[u];
          dst[j + half] = x2[u];
        }
      }
    } else {
      const int pos = p.pos[row];
      if (pos < 0) {
        if (lane == 0) atomicOr(p.status, 0x2u);
        continue;
      }
      const int slot = pos % p.window;
      const size_t off =
          ((((size_t)layer * 2 + (kind == 2)) * p.n_head_kv + head) * p.window + slot) * hd;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = lane + 32 * u;
        if (j >= half) continue;
        if (p.ring_bf16) {
          uint16_t* d = reinterpret_cast<uint16_t*>(p.ring_seq) + off;
          d[j] = f32_to_bf16_bits(x1[u]);
          d[j + half] = f32_to_bf16_bits(x2[u]);
        } else {
          float* d = reinterpret_cast<float*>(p.ring_seq) + off;
          d[j] = x1[u];
          d[j + half] = x2[u];
        }
      }
    }
  }
}

// ------------------------------------------------------------------ kernel

// Stream-K schedule: the work is n_items = n_tiles x n_mb output tiles (128
// weight rows x 16 activation rows), each cut into cpt chunks along k.  The
// grid is one resident wave; CTA b owns units [U b / G, U (b+1) / G) of the
// U = n_items * cpt units in item-major order, so every CTA streams the same
// number of weight bytes and there is no tail wave.  A tile finished inside one
// CTA goes straight to the epilogue; a tile shared by several CTAs is summed by
// the last of them (atomic ticket) in CTA order, which keeps results
// deterministic.  CTA c keeps at most two partial tiles: slot 2c for the tile
// its range starts inside, slot 2c + 1 for the tile its range ends inside.
DF_DEVICE long long owner_of(long long u, long long U, int G) { return ((u + 1) * G - 1) / U; }

template <int WT>
__global__ void __launch_bounds__(kGemmThreads) gemm_rows_kernel(const __grid_constant__ GemmParams p) {
  using T = WTraits<WT>;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_flag;
  const int XS = p.xk + T::PAD;
  uint16_t* xs_hi = reinterpret_cast<uint16_t*>(smem);
  uint16_t* xs_lo = xs_hi + 16 * XS;
  float* acc_s = reinterpret_cast<float*>(xs_lo + 16 * XS);
  float* inv_rms = acc_s + 16 * kTileRows;
  float* scale_s = inv_rms + 16;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int G = gridDim.x, b = blockIdx.x;
  const long long U = (long long)p.n_tiles * p.n_mb * p.cpt;
  const long long ub0 = U * b / G, ub1 = U * (b + 1) / G;
  const bool has_lo = p.x_mode != X_BF16;
  bool waited = false;
  pdl_trigger();

  for (long long u = ub0; u < ub1;) {
    const int item = (int)(u / p.cpt);
    const int c0 = (int)(u - (long long)item * p.cpt);
    const int c1 = (int)min((long long)p.cpt, c0 + (ub1 - u));
    u += c1 - c0;
    const int tile = item / p.n_mb, mb = item - tile * p.n_mb;
    const int m0 = mb * 16;

    __syncthreads();  // the previous segment is done with shared memory
    if (tid < kTileRows) {
      const float* sc = nullptr;
      const uint8_t* r = map_row(p, tile, tid, T::ESZ, &sc);
      scale_s[tid] = r ? (sc ? *sc : 1.f) : 0.f;
    }
    const float* dummy;
    const uint8_t* wa = map_row(p, tile, warp * 16 + g, T::ESZ, &dummy);
    const uint8_t* wb = map_row(p, tile, warp * 16 + g + 8, T::ESZ, &dummy);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int k0 = c0 * T::KC, k1 = c1 * T::KC;

    for (int xs0 = k0; xs0 < k1; xs0 += p.xk) {
      const int xlen = min(p.xk, k1 - xs0);
      const int nch = xlen / T::KC;
      const uint8_t* pa = wa ? wa + (size_t)(xs0 + T::EPL * t) * T::ESZ : nullptr;
      const uint8_t* pb = wb ? wb + (size_t)(xs0 + T::EPL * t) * T::ESZ : nullptr;
      uint4 ra[T::U][T::NV], rb[T::U][T::NV], na[T::U][T::NV], nb[T::U][T::NV];
      // weights do not depend on the activations: start streaming before staging x
      load_stage<WT>(ra, rb, pa, pb, 0, nch);
      if (!waited) {
        pdl_wait();  // everything below may read what earlier kernels wrote
        waited = true;
      }
      if (xs0 == k0 && tid < 16) {
        float inv = 1.f;
        if (p.normw && m0 + tid < p.M) {
          float sum = 0.f;
          for (int q = 0; q < p.n_ss; ++q) sum += p.ss[(size_t)q * p.ss_ld + m0 + tid];
          inv = 1.f / sqrtf(sum / (float)p.K + p.eps);
        }
        inv_rms[tid] = inv;
      }
      __syncthreads();
      stage_x(p, xs_hi, xs_lo, XS, inv_rms, m0, xs0, xlen);
      __syncthreads();
      for (int cc = 0; cc < nch; cc += 2 * T::U) {
        load_stage<WT>(na, nb, pa, pb, cc + T::U, nch);
        compute_stage<WT>(ra, rb, xs_hi, xs_lo, XS, cc, nch, g, t, has_lo, acc);
        if (cc + T::U >= nch) break;
        load_stage<WT>(ra, rb, pa, pb, cc + 2 * T::U, nch);
        compute_stage<WT>(na, nb, xs_hi, xs_lo, XS, cc + T::U, nch, g, t, has_lo, acc);
      }
    }

    // accumulators -> shared tile [act row][weight row]
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = 8 * j + 2 * t, r = warp * 16 + g;
      acc_s[c * kTileRows + r] = acc[j][0];
      acc_s[(c + 1) * kTileRows + r] = acc[j][1];
      acc_s[c * kTileRows + r + 8] = acc[j][2];
      acc_s[(c + 1) * kTileRows + r + 8] = acc[j][3];
    }
    __syncthreads();

    if (c0 != 0 || c1 != p.cpt) {
      const long long iu0 = (long long)item * p.cpt;
      const int first = (int)owner_of(iu0, U, G);
      const int last = (int)owner_of(iu0 + p.cpt - 1, U, G);
      const size_t slot = 2 * (size_t)b + (b == first ? 1 : 0);
      float* part = p.partial + slot * (16 * kTileRows);
      for (int i = tid; i < 16 * kTileRows; i += blockDim.x) part[i] = acc_s[i];
      __threadfence();
      __syncthreads();
      if (tid == 0) s_flag = atomicAdd(p.counters + item, 1) == last - first;
      __syncthreads();
      if (!s_flag) continue;
      __threadfence();
      for (int i = tid; i < 16 * kTileRows; i += blockDim.x) {
        float sum = 0.f;
        for (int c = first; c <= last; ++c) {
          const size_t sl = 2 * (size_t)c + (c == first ? 1 : 0);
          sum += __ldcg(p.partial + sl * (16 * kTileRows) + i);
        }
        acc_s[i] = sum;
      }
      if (tid == 0) p.counters[item] = 0;
      __syncthreads();
    }

    switch (p.epi) {
      case EPI_SWIGLU:
        epilogue_swiglu(p, acc_s, scale_s, mb, tile);
        break;
      case EPI_QKV:
      case EPI_INJECT:
        epilogue_heads(p, acc_s, scale_s, mb, tile);
        break;
      default:
        epilogue_rows(p, acc_s, scale_s, mb, tile, &s_flag);
        break;
    }
  }
}

cudaError_t configure_gemm(int xk_max) {
  cudaError_t e = cudaFuncSetAttribute(gemm_rows_kernel<W_F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gemm_smem_bytes(W_F32, xk_max));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_rows_kernel<W_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gemm_smem_bytes(W_BF16, xk_max));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_rows_kernel<W_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gemm_smem_bytes(W_FP8, xk_max));
  return e;
}

template <int WT>
static cudaError_t launch_t(const GemmParams& p, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(WT, p.xk);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_rows_kernel<WT>, p);
}

cudaError_t launch_gemm(int wt, const GemmParams& p, cudaStream_t st) {
  switch (wt) {
    case W_F32: return launch_t<W_F32>(p, st);
    case W_BF16: return launch_t<W_BF16>(p, st);
    case W_FP8: return launch_t<W_FP8>(p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dflash
