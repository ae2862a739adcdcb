// Sliding-window GQA attention of the noise block.
//
// The block's 16 rows at positions n_past .. n_past + 15 attend (non-causally)
// to every row of the block and to the ring slots holding positions p with
// 0 <= p < n_past and (n_past + i) - p < window (dflash-ops model card, Method).
// Every kernel here works on (sequence, kv head, group of query heads): the
// ring of the kv head is cut into 64-key sub-chunks staged into shared memory
// by async copies, warp (h, q) owns query head h of the group and key lane q,
// and key lane q attends to its sub-chunks with an online softmax, so the
// heads of the kv group share every K/V tile.  Both products use the tensor
// cores (mma.sync) with fp32 accumulation: q and the probabilities are split
// into bf16 hi + lo, bf16 ring K/V are exact, fp32 K/V (an fp32 ring, the
// block's own keys) are split too.  Partial (max, sum, O) states are merged in
// a fixed order, and the o projection's input is written as a 16-bit hi/lo
// pair.  Three launch forms (launch_attention picks one per step):
//   - split window (attn_split_kernel): every window in CTAs of 128 slots, the
//     whole grid resident at once, merged through global scratch - one or a
//     few sequences;
//   - stream-K (attn_stream_kernel + attn_plan_kernel): one CTA per SM over
//     equal ranges of all windows' non-empty sub-chunks - larger batches with
//     a bf16 ring and head_dim >= 64;
//   - clusters (attn_cluster_kernel): a window over the CTAs of a thread-block
//     cluster, merged through distributed shared memory - the remaining cases.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

#include <math_constants.h>

#include <algorithm>
#include <mutex>
#include <vector>

namespace cg = cooperative_groups;

namespace dflash {

constexpr int kSub = 64;       // keys per sub-chunk
constexpr int kPad = 8;        // bf16 row padding (conflict-free fragment loads)
constexpr int kMaxCluster = 8;
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = exp2(x log2 e)

DF_DEVICE uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
DF_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count) : "memory");
}
DF_DEVICE void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes)
               : "memory");
}
// Wait for the phase with this parity to complete; false after ~2 s.
DF_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(su32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > 4000000000LL) return false;
  }
}
// One contiguous global -> shared copy by the bulk-copy engine (16-byte
// aligned addresses, size a multiple of 16), completing on `bar`.
DF_DEVICE void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}

// CTA b of G's share of the attention's L2 prefetch range, in 16-byte aligned
// pieces of at most 32 KB (thread 0: the bulk prefetches take no registers).
DF_DEVICE void prefetch_share_attn(const AttnParams& p, long long b, long long G) {
  if (!p.pf_bytes) return;
  const unsigned long long x0 = (p.pf_bytes * b / G) & ~15ull;
  const unsigned long long x1 = b == G - 1 ? p.pf_bytes : (p.pf_bytes * (b + 1) / G) & ~15ull;
  for (unsigned long long x = x0; x < x1;) {
    unsigned long long n = x1 - x;
    if (n > 32768) n = 32768;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.pf_base + x), "r"((uint32_t)n) : "memory");
    x += n;
  }
}

DF_DEVICE void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}

DF_DEVICE void ldsm_x4(uint32_t (&r)[4], const void* smem) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
DF_DEVICE void ldsm_x4_t(uint32_t (&r)[4], const void* smem) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

// Launch plan: query heads per CTA (hpc, a divisor of the group size), key
// lanes per head (kq: warps per head; warps = hpc * kq <= 8) and staging
// buffers (nb 64-key sub-chunks in flight, a multiple of kq).
struct AttnPlan {
  int hpc, kq, nb;
};
// bf16 ring: four buffers stage a whole 256-key slice at once (one CTA per
// SM); fp32 ring: two, whose hi/lo tiles take twice the room.  The throughput
// plan of large batched grids stages two sub-chunks with four warps so that
// two CTAs share an SM and overlap one another's copies and math.
constexpr int kLatencyPlans = 4;
inline int plans_for(bool f32, int G, int n_sub, AttnPlan (&out)[kLatencyPlans + 1]) {
  const int nb_max = f32 ? 2 : 4;
  int n = 0;
  const int hpcs[3] = {4, 2, 1};
  const int kqs[3] = {4, 2, 1};
  for (int hpc : hpcs) {
    if (G % hpc) continue;
    for (int kq : kqs) {
      if (hpc * kq > 8 || kq > nb_max || hpc * kq < 4 || n >= kLatencyPlans) continue;
      // no more buffers than the slice has sub-chunks (rounded up to the key lanes)
      const int nb = std::min(nb_max, std::max(kq, (n_sub + kq - 1) / kq * kq));
      out[n++] = AttnPlan{hpc, kq, nb};
    }
  }
  if (n == 0) out[n++] = AttnPlan{1, nb_max, nb_max};  // groups of odd size
  int h2 = G % 2 == 0 ? 2 : 1;
  out[n++] = AttnPlan{h2, 2, 2};               // throughput plan (last)
  return n;
}

template <int HD>
struct AttnSmem {
  static constexpr int KS = HD + kPad;
  static constexpr int TILE = kSub * KS;               // one [64][KS] bf16 tile (elements)
  // a bf16 ring with hd >= 64 is staged by TMA: [64 slots][HD] tiles of 64-dim
  // boxes, 128-byte swizzled (no padding), the buffers 1024-byte aligned
  static constexpr bool kTma = HD >= 64;
  static constexpr int TILE_SW = kSub * HD;
  // buffer b: K hi, V hi, K lo, V lo (lo only used by an fp32 ring)
  static constexpr int BUF = 4 * TILE;
  static constexpr int BLK = 4 * kBlock * KS;          // block keys: K hi/lo, V hi/lo [16][KS]
  // staging: nb sub-chunk buffers, the block keys, nb x 64 slot positions
  static constexpr __host__ __device__ size_t buf_elems(bool f32) {
    return f32 ? BUF : (kTma ? 2 * TILE_SW : 2 * TILE);
  }
  static size_t stage_bytes(bool f32, int nb) {
    return (size_t)nb * buf_elems(f32) * 2 + (size_t)BLK * 2 + (size_t)nb * kSub * 4;
  }
  // merge: per-warp fragments [warps][HD/8][32] float4 + (m, l) float4 per lane,
  // then the CTA's partial [R][HD] + (m, l)
  static size_t merge_bytes(int warps, int R) {
    return (size_t)warps * (HD / 8) * 32 * 16 + (size_t)warps * 32 * 16 + (size_t)R * HD * 4 +
           (size_t)R * 8;
  }
  static size_t bytes(bool f32, const AttnPlan& pl) {
    const size_t a = stage_bytes(f32, pl.nb) + (kTma && !f32 ? 1024 : 0),
                 b = merge_bytes(pl.kq * pl.hpc, kBlock * pl.hpc);
    return (a > b ? a : b) + 256;
  }
};

// Online-softmax update of one warp's 16 rows with one tile of up to 64 keys.
// element offset of (row, dim) in a swizzled [64][HD] ring tile: 64-dim boxes of
// 64 rows x 128 bytes, 16-byte chunk c of row r at chunk c ^ (r % 8)
template <int HD>
DF_DEVICE int sw_off(int row, int dim) {
  return (dim >> 6) * (kSub * 64) + row * 64 + ((((dim & 63) >> 3) ^ (row & 7)) << 3);
}

template <int HD, bool SPLIT, bool SW = false>
DF_DEVICE void attend_tile(const uint32_t (&qh)[HD / 16][4], const uint32_t (&ql)[HD / 16][4],
                           const uint16_t* k_hi, const uint16_t* k_lo, const uint16_t* v_hi,
                           const uint16_t* v_lo, int KS, int nt, const int* kpos, bool blk, int p0,
                           int window, int bw, float& m0, float& m1, float& l0, float& l1,
                           float (&O)[HD / 8][4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  float S[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
  // Key tiles in groups of four: the hi-q products of the group, then its lo-q
  // products, so that the two updates of an accumulator are four MMAs apart
  const int lm = lane >> 3;
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
    for (int j0 = 0; j0 < 8; j0 += 4) {
      if (j0 < nt) {
        // B fragments of key tiles j and j + 1 (k = dims ks*16 .. +15) in one
        // ldmatrix: lane i addresses key 8 (j + i/16) + i%8, dims + 8 ((i/8)%2)
        uint32_t b[2][4];
        int off[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int row = 8 * (j0 + 2 * u + (lm >> 1)) + (lane & 7), dim = ks * 16 + (lm & 1) * 8;
          off[u] = SW ? sw_off<HD>(row, dim) : row * KS + dim;
          if (j0 + 2 * u < nt) ldsm_x4(b[u], k_hi + off[u]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (j0 + 2 * u < nt) {
            mma_bf16_16816(S[j0 + 2 * u], qh[ks], b[u][0], b[u][1]);
            mma_bf16_16816(S[j0 + 2 * u + 1], qh[ks], b[u][2], b[u][3]);
          }
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (j0 + 2 * u < nt) {
            mma_bf16_16816(S[j0 + 2 * u], ql[ks], b[u][0], b[u][1]);
            mma_bf16_16816(S[j0 + 2 * u + 1], ql[ks], b[u][2], b[u][3]);
          }
        if (SPLIT) {
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (j0 + 2 * u < nt) ldsm_x4(b[u], k_lo + off[u]);
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (j0 + 2 * u < nt) {
              mma_bf16_16816(S[j0 + 2 * u], qh[ks], b[u][0], b[u][1]);
              mma_bf16_16816(S[j0 + 2 * u + 1], qh[ks], b[u][2], b[u][3]);
            }
        }
      }
    }
  }
  // mask; tile row max
  const int q0 = p0 + g, q1 = p0 + g + 8;
  float t0 = -CUDART_INF_F, t1 = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        bool ok0 = true, ok1 = true;
        if (blk) {  // block keys past the block's width do not exist
          ok0 = ok1 = 8 * j + 2 * t + e < bw;
        } else {
          const int kp = kpos[8 * j + 2 * t + e];
          const bool past = kp >= 0 && kp < p0;
          ok0 = past && q0 - kp < window;
          ok1 = past && q1 - kp < window;
        }
        if (!ok0) S[j][e] = -CUDART_INF_F;
        if (!ok1) S[j][2 + e] = -CUDART_INF_F;
        t0 = fmaxf(t0, S[j][e]);
        t1 = fmaxf(t1, S[j][2 + e]);
      }
    }
  }
  t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, 1));
  t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, 2));
  t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, 1));
  t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, 2));
  const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
  // rescale the running sums to the new maxima (nothing to rescale while -inf)
  const float c0 = m0 == -CUDART_INF_F ? 0.f : exp2f(m0 - n0);
  const float c1 = m1 == -CUDART_INF_F ? 0.f : exp2f(m1 - n1);
  m0 = n0;
  m1 = n1;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        S[j][e] = n0 == -CUDART_INF_F ? 0.f : exp2f(S[j][e] - n0);
        S[j][2 + e] = n1 == -CUDART_INF_F ? 0.f : exp2f(S[j][2 + e] - n1);
        s0 += S[j][e];
        s1 += S[j][2 + e];
      }
    } else {
      S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
    }
  }
  s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
  s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
  l0 = l0 * c0 + s0;
  l1 = l1 * c1 + s1;
#pragma unroll
  for (int jd = 0; jd < HD / 8; ++jd) {
    O[jd][0] *= c0;
    O[jd][1] *= c0;
    O[jd][2] *= c1;
    O[jd][3] *= c1;
  }
  uint32_t ph[4][4], pl[4][4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    split_bf16x2(S[2 * kk][0], S[2 * kk][1], ph[kk][0], pl[kk][0]);
    split_bf16x2(S[2 * kk][2], S[2 * kk][3], ph[kk][1], pl[kk][1]);
    split_bf16x2(S[2 * kk + 1][0], S[2 * kk + 1][1], ph[kk][2], pl[kk][2]);
    split_bf16x2(S[2 * kk + 1][2], S[2 * kk + 1][3], ph[kk][3], pl[kk][3]);
  }
  // output dims in groups of four n8 tiles: per 16-key step the hi-p products
  // of the group, then its lo-p products (accumulator updates four MMAs apart)
  const int lrow = lane & 7, lmat = lane >> 3;
#pragma unroll
  for (int jd = 0; jd < HD / 8; jd += 4) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (2 * kk < nt) {
        const int key = 16 * kk + (lmat & 1) * 8 + lrow;
        uint32_t b[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int dim = 8 * (jd + 2 * u) + (lmat >> 1) * 8;
          ldsm_x4_t(b[u], v_hi + (SW ? sw_off<HD>(key, dim) : key * KS + dim));
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          mma_bf16_16816(O[jd + 2 * u], ph[kk], b[u][0], b[u][1]);
          mma_bf16_16816(O[jd + 2 * u + 1], ph[kk], b[u][2], b[u][3]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          mma_bf16_16816(O[jd + 2 * u], pl[kk], b[u][0], b[u][1]);
          mma_bf16_16816(O[jd + 2 * u + 1], pl[kk], b[u][2], b[u][3]);
        }
        if (SPLIT) {
#pragma unroll
          for (int u = 0; u < 2; ++u)
            ldsm_x4_t(b[u], v_lo + key * KS + 8 * (jd + 2 * u) + (lmat >> 1) * 8);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            mma_bf16_16816(O[jd + 2 * u], ph[kk], b[u][0], b[u][1]);
            mma_bf16_16816(O[jd + 2 * u + 1], ph[kk], b[u][2], b[u][3]);
          }
        }
      }
    }
  }
}

// Cluster kernel: one thread-block cluster per (sequence, kv head, group of
// query heads); the ring of the kv head is split between the CL CTAs of the
// cluster, each CTA stages its slots' sub-chunks nb at a time (a round) and
// key lane q attends to sub-chunk q of each round as soon as it lands.  The
// key lanes merge inside the CTA, then the cluster's CTAs merge through
// distributed shared memory in rank order; rank 0 also attends to the block's
// own keys.
template <int HD, bool RING_F32>
__global__ void __launch_bounds__(256) attn_cluster_kernel(const __grid_constant__ AttnParams p) {
  using SM = AttnSmem<HD>;
  constexpr int KS = SM::KS;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const int G = p.n_head / p.n_head_kv, hpc = p.hpc, kq = p.kq, nb = p.nb, n_hgrp = G / hpc;
  const int kvh = blockIdx.y / n_hgrp, hgrp = blockIdx.y - kvh * n_hgrp, seq = blockIdx.z;
  const int R = kBlock * hpc;                       // rows of this CTA (head-major)
  const int head0 = kvh * G + hgrp * hpc;           // first query head of the CTA
  const int qd = p.n_head * HD, kvd = p.n_head_kv * HD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int nwarps = (int)(blockDim.x >> 5);
  const int hl = warp / kq, lk = warp - hl * kq;    // head within the CTA, key lane
  constexpr bool TMA = !RING_F32 && SM::kTma;
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint16_t* bufs = reinterpret_cast<uint16_t*>(
      TMA ? (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023) : reinterpret_cast<uintptr_t>(sm_raw));
  const int buf_elems = (int)SM::buf_elems(RING_F32);
  uint16_t* blk_k_hi = bufs + nb * buf_elems;
  uint16_t* blk_k_lo = blk_k_hi + kBlock * KS;
  uint16_t* blk_v_hi = blk_k_lo + kBlock * KS;
  uint16_t* blk_v_lo = blk_v_hi + kBlock * KS;
  int* kpos = reinterpret_cast<int*>(blk_v_lo + kBlock * KS);  // [nb][64]
  __shared__ __align__(8) uint64_t s_bar[4];                    // one per staging buffer

  if (!RING_F32 && tid == 0) {
    for (int b = 0; b < nb; ++b) mbar_init(&s_bar[b], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid == 0) stamp_begin(p.stamp);
  __syncthreads();
  pdl_trigger();
  pdl_wait();
  const int p0 = max(p.n_past[seq], 0);
  const int per = (p.window + CL - 1) / CL;
  const int s_begin = min(p.window, rank * per), s_end = min(p.window, s_begin + per);
  const int n_sub = (s_end - s_begin + kSub - 1) / kSub;
  const size_t plane = (size_t)p.window * HD;
  const size_t kbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 0) * p.n_head_kv + kvh) * plane;
  const size_t vbase = kbase + (size_t)p.n_head_kv * plane;

  // Stage the ring rows of the round of sub-chunks j0 .. j0 + nb - 1 (buffer
  // j % nb).  A bf16 ring row (hd bf16, 16-byte aligned in both spaces) is one
  // bulk copy that completes on the buffer's mbarrier; rows past the CTA's
  // slots are zeroed.  An fp32 ring is loaded and split into bf16 hi/lo by the
  // threads.
  auto stage_round = [&](int j0) {
    const int jn = min(n_sub, j0 + nb);
    if (TMA) {
      // per sub-chunk: K and V as HD/64 boxes of 64 slots x 64 dims each (slots
      // past the CTA's range are the next ones in memory or the zero fill past
      // the ring: finite, and masked by their slot position)
      __syncthreads();  // earlier reads of the buffers are done
      if (tid == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const int row_k = (int)(kbase / HD), row_v = (int)(vbase / HD);
        for (int j = j0; j < jn; ++j) {
          mbar_expect_tx(&s_bar[j % nb], (uint32_t)(2 * SM::TILE_SW * 2));
          uint16_t* dst = bufs + (j % nb) * buf_elems;
          const int s0 = s_begin + j * kSub;
#pragma unroll
          for (int kv = 0; kv < 2; ++kv)
#pragma unroll
            for (int hb = 0; hb < HD / 64; ++hb)
              tma_load_2d(dst + kv * SM::TILE_SW + hb * kSub * 64, &p.tm_ring, hb * 64,
                          (kv ? row_v : row_k) + s0, &s_bar[j % nb]);
        }
      }
    } else if (!RING_F32) {
      if (tid == 0)
        for (int j = j0; j < jn; ++j) {
          const int nk = min(kSub, s_end - (s_begin + j * kSub));
          mbar_expect_tx(&s_bar[j % nb], (uint32_t)nk * HD * 2 * 2);
        }
      __syncthreads();  // expectations first; earlier reads of the buffers are done
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint16_t* r = reinterpret_cast<const uint16_t*>(p.ring);
      for (int idx = tid; idx < (jn - j0) * 2 * kSub; idx += blockDim.x) {
        const int jj = idx / (2 * kSub), rem = idx - jj * 2 * kSub;
        const int kv = rem / kSub, row = rem - kv * kSub, j = j0 + jj;
        const int s0 = s_begin + j * kSub, nk = min(kSub, s_end - s0);
        uint16_t* dst = bufs + (j % nb) * buf_elems + kv * SM::TILE + row * KS;
        if (row < nk) {
          bulk_copy(dst, r + (kv ? vbase : kbase) + (size_t)(s0 + row) * HD, HD * 2, &s_bar[j % nb]);
        } else {
#pragma unroll
          for (int d = 0; d < HD; d += 8) *reinterpret_cast<uint4*>(dst + d) = make_uint4(0, 0, 0, 0);
        }
      }
    } else {
      const float* r = reinterpret_cast<const float*>(p.ring);
      for (int j = j0; j < jn; ++j) {
        uint16_t* kh = bufs + (j % nb) * buf_elems;
        uint16_t* vh = kh + SM::TILE;
        uint16_t* kl = vh + SM::TILE;
        uint16_t* vl = kl + SM::TILE;
        const int s0 = s_begin + j * kSub, nk = min(kSub, s_end - s0);
        for (int idx = tid; idx < kSub * (HD / 4); idx += blockDim.x) {
          const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
          float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
          if (row < nk) {
            kv = *reinterpret_cast<const float4*>(r + kbase + (size_t)(s0 + row) * HD + d);
            vv = *reinterpret_cast<const float4*>(r + vbase + (size_t)(s0 + row) * HD + d);
          }
          uint2 h, l;
          split_bf16x2(kv.x, kv.y, h.x, l.x);
          split_bf16x2(kv.z, kv.w, h.y, l.y);
          *reinterpret_cast<uint2*>(kh + row * KS + d) = h;
          *reinterpret_cast<uint2*>(kl + row * KS + d) = l;
          split_bf16x2(vv.x, vv.y, h.x, l.x);
          split_bf16x2(vv.z, vv.w, h.y, l.y);
          *reinterpret_cast<uint2*>(vh + row * KS + d) = h;
          *reinterpret_cast<uint2*>(vl + row * KS + d) = l;
        }
      }
    }
  };
  // slot positions of the round's sub-chunks (-1 past the CTA's slots), at
  // most kPosPer per thread, all loads issued before the stores
  constexpr int kPosPer = 4;
  auto stage_kpos = [&](int j0) {
    const int n = (min(n_sub, j0 + nb) - j0) * kSub;
    for (int base = 0; base < n; base += kPosPer * (int)blockDim.x) {
      int v[kPosPer];
#pragma unroll
      for (int u = 0; u < kPosPer; ++u) {
        const int idx = base + u * (int)blockDim.x + tid;
        const int jj = idx / kSub, row = idx - jj * kSub, s0 = s_begin + (j0 + jj) * kSub;
        v[u] = idx < n && s0 + row < s_end ? p.ring_pos[(size_t)seq * p.window + s0 + row] : -1;
      }
#pragma unroll
      for (int u = 0; u < kPosPer; ++u) {
        const int idx = base + u * (int)blockDim.x + tid;
        const int jj = idx / kSub, row = idx - jj * kSub;
        if (idx < n) kpos[((j0 + jj) % nb) * kSub + row] = v[u];
      }
    }
  };
  // wait for the bulk copies of sub-chunk j (round r is its buffer's r-th phase)
  auto wait_sub = [&](int j, int r) {
    if (RING_F32) return;
    if (!mbar_wait(&s_bar[j % nb], (uint32_t)(r & 1))) {
      if (lane == 0) atomicOr(p.status, 0x4u);
      mbar_wait(&s_bar[j % nb], (uint32_t)(r & 1));  // a second bounded wait before moving on
    }
  };

  // the first round's copies go out before anything else; then one batch of
  // independent loads (q rows, the block's own keys, the round's slot
  // positions) whose values are consumed only after all of them are issued
  stage_round(0);
  const bool active = hl < hpc;
  float2 qraw[HD / 16][4];
  if (active) {
    const float* qr0 = p.q + (size_t)(seq * kBlock + g) * qd + (head0 + hl) * HD;
    const float* qr1 = qr0 + (size_t)8 * qd;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const int k0 = ks * 16 + 2 * t;
      qraw[ks][0] = *reinterpret_cast<const float2*>(qr0 + k0);
      qraw[ks][1] = *reinterpret_cast<const float2*>(qr1 + k0);
      qraw[ks][2] = *reinterpret_cast<const float2*>(qr0 + k0 + 8);
      qraw[ks][3] = *reinterpret_cast<const float2*>(qr1 + k0 + 8);
    }
  }
  if (rank == 0) {  // the block's own 16 keys (fp32: split hi/lo), <= 4 float4 per thread a pass
    constexpr int kBlkPer = 4, n = kBlock * (HD / 4);
    for (int base = 0; base < n; base += kBlkPer * (int)blockDim.x) {
      float4 kr[kBlkPer], vr[kBlkPer];
#pragma unroll
      for (int u = 0; u < kBlkPer; ++u) {
        const int idx = base + u * (int)blockDim.x + tid;
        kr[u] = vr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < n) {
          const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
          const size_t o = (size_t)(seq * kBlock + row) * kvd + kvh * HD + d;
          kr[u] = *reinterpret_cast<const float4*>(p.kblk + o);
          vr[u] = *reinterpret_cast<const float4*>(p.vblk + o);
        }
      }
#pragma unroll
      for (int u = 0; u < kBlkPer; ++u) {
        const int idx = base + u * (int)blockDim.x + tid;
        if (idx >= n) continue;
        const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
        uint2 h, l;
        split_bf16x2(kr[u].x, kr[u].y, h.x, l.x);
        split_bf16x2(kr[u].z, kr[u].w, h.y, l.y);
        *reinterpret_cast<uint2*>(blk_k_hi + row * KS + d) = h;
        *reinterpret_cast<uint2*>(blk_k_lo + row * KS + d) = l;
        split_bf16x2(vr[u].x, vr[u].y, h.x, l.x);
        split_bf16x2(vr[u].z, vr[u].w, h.y, l.y);
        *reinterpret_cast<uint2*>(blk_v_hi + row * KS + d) = h;
        *reinterpret_cast<uint2*>(blk_v_lo + row * KS + d) = l;
      }
    }
  }
  stage_kpos(0);
  // this warp's head: q fragments scaled by log2(e)/sqrt(hd) (scores in base-2
  // units: softmax weights are exp2(s - max)), split into bf16 hi/lo
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
  const float qscale = p.scale * kLog2e;
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      split_bf16x2(qraw[ks][e].x * qscale, qraw[ks][e].y * qscale, qh[ks][e], ql[ks][e]);
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float O[HD / 8][4];
#pragma unroll
  for (int jd = 0; jd < HD / 8; ++jd) O[jd][0] = O[jd][1] = O[jd][2] = O[jd][3] = 0.f;
  // the block's own keys go to the key lane with the least ring work, first:
  // their tile overlaps the wait for the ring copies
  const bool blk_lane = rank == 0 && active && lk == n_sub % kq;

  // rounds of nb sub-chunks; key lane q takes sub-chunks q, q + kq, ... of each
  // round, each as soon as its own copies have landed
  for (int j0 = 0, r = 0; j0 < n_sub; j0 += nb, ++r) {
    if (j0 > 0) {
      stage_round(j0);
      stage_kpos(j0);
    }
    __syncthreads();  // zeroed rows, slot positions, fp32 tiles and the block keys
    if (j0 == 0 && blk_lane)
      attend_tile<HD, true>(qh, ql, blk_k_hi, blk_k_lo, blk_v_hi, blk_v_lo, KS, 2, nullptr, true,
                            p0, p.window, p.block_width, m0, m1, l0, l1, O, lane);
    for (int j = j0 + lk; j < min(n_sub, j0 + nb); j += kq) {
      wait_sub(j, r);
      // row 0 has the widest window: a sub-chunk with no key for it has none
      // for any row (empty slots of a partly filled ring, or out of window)
      const int* kp = kpos + (j % nb) * kSub;
      const int ka = kp[lane], kb = kp[lane + 32];
      const bool any = __any_sync(0xffffffffu, (ka >= 0 && ka < p0 && p0 - ka < p.window) ||
                                                   (kb >= 0 && kb < p0 && p0 - kb < p.window));
      if (active && any) {
        const uint16_t* kh = bufs + (j % nb) * buf_elems;
        if (TMA)
          attend_tile<HD, false, true>(qh, ql, kh, nullptr, kh + SM::TILE_SW, nullptr, KS, 8,
                                       kpos + (j % nb) * kSub, false, p0, p.window, 16, m0, m1, l0,
                                       l1, O, lane);
        else
          attend_tile<HD, RING_F32>(qh, ql, kh, kh + 2 * SM::TILE, kh + SM::TILE, kh + 3 * SM::TILE,
                                    KS, 8, kpos + (j % nb) * kSub, false, p0, p.window, 16, m0, m1, l0,
                                    l1, O, lane);
      }
    }
    __syncthreads();  // the buffers are restaged by the next round
  }
  if (n_sub == 0) {   // a CTA with no ring slots
    __syncthreads();
    if (blk_lane)
      attend_tile<HD, true>(qh, ql, blk_k_hi, blk_k_lo, blk_v_hi, blk_v_lo, KS, 2, nullptr, true,
                            p0, p.window, p.block_width, m0, m1, l0, l1, O, lane);
    __syncthreads();
  }

  // 1. key lanes 1.. of each head hand their (max, sum, O) fragments to key
  //    lane 0 through shared memory (over the staging buffers), which merges
  //    them into its registers in lane order
  float4* frag_o = reinterpret_cast<float4*>(sm_raw);                     // [warps][HD/8][32]
  float4* frag_ml = frag_o + (size_t)nwarps * (HD / 8) * 32;              // [warps][32]
  float* part_o = reinterpret_cast<float*>(frag_ml + (size_t)nwarps * 32);  // [R][HD]
  float2* part_ml = reinterpret_cast<float2*>(part_o + (size_t)R * HD);   // [R]
  if (active && lk > 0) {
#pragma unroll
    for (int jd = 0; jd < HD / 8; ++jd)
      frag_o[((size_t)warp * (HD / 8) + jd) * 32 + lane] = make_float4(O[jd][0], O[jd][1], O[jd][2], O[jd][3]);
    frag_ml[warp * 32 + lane] = make_float4(m0, m1, l0, l1);
  }
  __syncthreads();
  if (active && lk == 0) {
    for (int q = 1; q < kq; ++q) {
      const int w = warp + q;
      const float4 ml = frag_ml[w * 32 + lane];
      const float n0 = fmaxf(m0, ml.x), n1 = fmaxf(m1, ml.y);
      const float a0 = m0 == -CUDART_INF_F ? 0.f : exp2f(m0 - n0);
      const float b0 = ml.x == -CUDART_INF_F ? 0.f : exp2f(ml.x - n0);
      const float a1 = m1 == -CUDART_INF_F ? 0.f : exp2f(m1 - n1);
      const float b1 = ml.y == -CUDART_INF_F ? 0.f : exp2f(ml.y - n1);
      m0 = n0;
      m1 = n1;
      l0 = a0 * l0 + b0 * ml.z;
      l1 = a1 * l1 + b1 * ml.w;
#pragma unroll
      for (int jd = 0; jd < HD / 8; ++jd) {
        const float4 v = frag_o[((size_t)w * (HD / 8) + jd) * 32 + lane];
        O[jd][0] = a0 * O[jd][0] + b0 * v.x;
        O[jd][1] = a0 * O[jd][1] + b0 * v.y;
        O[jd][2] = a1 * O[jd][2] + b1 * v.z;
        O[jd][3] = a1 * O[jd][3] + b1 * v.w;
      }
    }
    // 2. this CTA's partial of the head's 16 rows, row-major for the peers
    float* o0 = part_o + (size_t)(hl * kBlock + g) * HD;
    float* o1 = o0 + (size_t)8 * HD;
#pragma unroll
    for (int jd = 0; jd < HD / 8; ++jd) {
      *reinterpret_cast<float2*>(o0 + 8 * jd + 2 * t) = make_float2(O[jd][0], O[jd][1]);
      *reinterpret_cast<float2*>(o1 + 8 * jd + 2 * t) = make_float2(O[jd][2], O[jd][3]);
    }
    if (t == 0) {
      part_ml[hl * kBlock + g] = make_float2(m0, l0);
      part_ml[hl * kBlock + g + 8] = make_float2(m1, l1);
    }
  }
  // 3. merge the cluster's CTAs through distributed shared memory, rank order
  cluster.sync();
  const int rows_per = (R + CL - 1) / CL;
  const int r_lo = rank * rows_per, r_hi = min(R, r_lo + rows_per);
  for (int r = r_lo + warp; r < r_hi; r += nwarps) {
    // remote loads first: lane c < CL fetches rank c's (max, sum), every lane
    // the ranks' partial O at its four dims (one round trip for both)
    const int d = lane * 4;
    float4 v[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c)
      v[c] = c < CL && d < HD
                 ? *reinterpret_cast<const float4*>(cluster.map_shared_rank(part_o, c) + (size_t)r * HD + d)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    float2 ml = make_float2(-CUDART_INF_F, 0.f);
    if (lane < CL) ml = cluster.map_shared_rank(part_ml, lane)[r];
    float M = ml.x;
#pragma unroll
    for (int o = kMaxCluster / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wgt = (lane < CL && ml.x != -CUDART_INF_F) ? exp2f(ml.x - M) : 0.f;
    float L = wgt * ml.y;
#pragma unroll
    for (int o = kMaxCluster / 2; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    L = __shfl_sync(0xffffffffu, L, 0);  // lanes 0..7 hold the total
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      const float wc = __shfl_sync(0xffffffffu, wgt, c);  // ranks summed in rank order
      acc.x += wc * v[c].x;
      acc.y += wc * v[c].y;
      acc.z += wc * v[c].z;
      acc.w += wc * v[c].w;
    }
    if (d < HD) {
      const int h = r / kBlock, i = r - h * kBlock;
      const float inv = 1.f / L;
      const size_t at = (size_t)(seq * kBlock + i) * qd + (head0 + h) * HD + d;
      uint2 hi, lo;
      split_pair16x2(acc.x * inv, acc.y * inv, p.pair_f16 != 0, hi.x, lo.x);
      split_pair16x2(acc.z * inv, acc.w * inv, p.pair_f16 != 0, hi.y, lo.y);
      *reinterpret_cast<uint2*>(p.out_hi + at) = hi;
      *reinterpret_cast<uint2*>(p.out_lo + at) = lo;
    }
  }
  cluster.sync();  // peers may still be reading this CTA's partials
  if (tid == 0) stamp_finish(p.stamp);
}

// ---------------------------------------------------------------------------
// Split-window attention (grids that the GPU holds at once).
//
// The cluster kernel above caps a kv head's window at kMaxCluster CTAs, and a
// cluster of 8 must find 8 free SMs in one GPC: one sequence of the real drafter
// (8 kv heads) ran on 64 of the 152 SMs.  Here the window of a (sequence, kv
// head, head group) is split into n_split independent CTAs of kq x 64 slots,
// one 64-key sub-chunk per key lane (one staging round), so the whole GPU
// works on one sequence.  Split 0 also attends to the block's 16 keys.  A CTA
// merges its key lanes in shared memory and publishes its partial rows - the
// running max m, the sum l and the un-normalised O of each query row - to
// global scratch, then arrives on its group's counter.  Once all n_split CTAs
// of the group have arrived (a wait bounded by ~2 s: the launcher uses this
// kernel only when the whole grid is resident at once, so every CTA of the
// group runs), CTA s merges rows s, s + n_split, ... of the group - weights
// exp2(m_c - max m) summed over the splits in split order, so results do not
// depend on arrival order - and writes the o projection's input pair.  The
// group's last CTA to finish its merge resets the two counters for the next
// launch.
// ---------------------------------------------------------------------------

constexpr int kMaxSplit = 32;   // splits per window (one lane each in the merge)

DF_DEVICE int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
DF_DEVICE int atom_add_release_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
DF_DEVICE int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

template <int HD, bool RING_F32>
__global__ void __launch_bounds__(256, 1) attn_split_kernel(const __grid_constant__ AttnParams p) {
  using SM = AttnSmem<HD>;
  constexpr int KS = SM::KS;
  const int G = p.n_head / p.n_head_kv, hpc = p.hpc, kq = p.kq, n_hgrp = G / hpc;
  const int split = blockIdx.x, n_split = gridDim.x;
  const int kvh = blockIdx.y / n_hgrp, hg = blockIdx.y - kvh * n_hgrp, seq = blockIdx.z;
  const int group = (seq * p.n_head_kv + kvh) * n_hgrp + hg;
  const int R = kBlock * hpc;                       // rows of this CTA (head-major)
  const int head0 = kvh * G + hg * hpc;             // first query head of the CTA
  const int qd = p.n_head * HD, kvd = p.n_head_kv * HD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int nwarps = (int)(blockDim.x >> 5);
  const int hl = warp / kq, lk = warp - hl * kq;    // head within the CTA, key lane
  constexpr bool TMA = !RING_F32 && SM::kTma;
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint16_t* bufs = reinterpret_cast<uint16_t*>(
      TMA ? (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023) : reinterpret_cast<uintptr_t>(sm_raw));
  const int buf_elems = (int)SM::buf_elems(RING_F32);
  uint16_t* blk_k_hi = bufs + kq * buf_elems;
  uint16_t* blk_k_lo = blk_k_hi + kBlock * KS;
  uint16_t* blk_v_hi = blk_k_lo + kBlock * KS;
  uint16_t* blk_v_lo = blk_v_hi + kBlock * KS;
  int* kpos = reinterpret_cast<int*>(blk_v_lo + kBlock * KS);  // [kq][64]
  __shared__ __align__(8) uint64_t s_bar[4];                    // one per sub-chunk buffer
  __shared__ int s_last;

  if (!RING_F32 && tid == 0) {
    for (int b = 0; b < kq; ++b) mbar_init(&s_bar[b], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid == 0) stamp_begin(p.stamp);
  __syncthreads();
  pdl_trigger();
  // the ring, its slot positions and n_past were written before the step's
  // first kernel (launched without overlap): they are read, and the ring staged,
  // before the wait for the q/k/v kernel
  const int p0 = max(p.n_past[seq], 0);
  const int SL = kq * kSub;
  const int s_begin = min(p.window, split * SL), s_end = min(p.window, s_begin + SL);
  const int n_sub = (s_end - s_begin + kSub - 1) / kSub;
  const size_t plane = (size_t)p.window * HD;
  const size_t kbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 0) * p.n_head_kv + kvh) * plane;
  const size_t vbase = kbase + (size_t)p.n_head_kv * plane;

  // stage sub-chunk j of the split into buffer j (the only round)
  if (TMA) {
    if (tid == 0) {
      const int row_k = (int)(kbase / HD), row_v = (int)(vbase / HD);
      for (int j = 0; j < n_sub; ++j) {
        mbar_expect_tx(&s_bar[j], (uint32_t)(2 * SM::TILE_SW * 2));
        uint16_t* dst = bufs + j * buf_elems;
        const int s0 = s_begin + j * kSub;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int hb = 0; hb < HD / 64; ++hb)
            tma_load_2d(dst + kv * SM::TILE_SW + hb * kSub * 64, &p.tm_ring, hb * 64,
                        (kv ? row_v : row_k) + s0, &s_bar[j]);
      }
    }
  } else if (!RING_F32) {
    if (tid == 0)
      for (int j = 0; j < n_sub; ++j) {
        const int nk = min(kSub, s_end - (s_begin + j * kSub));
        mbar_expect_tx(&s_bar[j], (uint32_t)nk * HD * 2 * 2);
      }
    __syncthreads();  // expectations before any copy can complete
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint16_t* r = reinterpret_cast<const uint16_t*>(p.ring);
    for (int idx = tid; idx < n_sub * 2 * kSub; idx += blockDim.x) {
      const int j = idx / (2 * kSub), rem = idx - j * 2 * kSub;
      const int kv = rem / kSub, row = rem - kv * kSub;
      const int s0 = s_begin + j * kSub, nk = min(kSub, s_end - s0);
      uint16_t* dst = bufs + j * buf_elems + kv * SM::TILE + row * KS;
      if (row < nk) {
        bulk_copy(dst, r + (kv ? vbase : kbase) + (size_t)(s0 + row) * HD, HD * 2, &s_bar[j]);
      } else {
#pragma unroll
        for (int d = 0; d < HD; d += 8) *reinterpret_cast<uint4*>(dst + d) = make_uint4(0, 0, 0, 0);
      }
    }
  } else {
    const float* r = reinterpret_cast<const float*>(p.ring);
    for (int j = 0; j < n_sub; ++j) {
      uint16_t* kh = bufs + j * buf_elems;
      uint16_t* vh = kh + SM::TILE;
      uint16_t* kl = vh + SM::TILE;
      uint16_t* vl = kl + SM::TILE;
      const int s0 = s_begin + j * kSub, nk = min(kSub, s_end - s0);
      for (int idx = tid; idx < kSub * (HD / 4); idx += blockDim.x) {
        const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
        float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
        if (row < nk) {
          kv = *reinterpret_cast<const float4*>(r + kbase + (size_t)(s0 + row) * HD + d);
          vv = *reinterpret_cast<const float4*>(r + vbase + (size_t)(s0 + row) * HD + d);
        }
        uint2 h, l;
        split_bf16x2(kv.x, kv.y, h.x, l.x);
        split_bf16x2(kv.z, kv.w, h.y, l.y);
        *reinterpret_cast<uint2*>(kh + row * KS + d) = h;
        *reinterpret_cast<uint2*>(kl + row * KS + d) = l;
        split_bf16x2(vv.x, vv.y, h.x, l.x);
        split_bf16x2(vv.z, vv.w, h.y, l.y);
        *reinterpret_cast<uint2*>(vh + row * KS + d) = h;
        *reinterpret_cast<uint2*>(vl + row * KS + d) = l;
      }
    }
  }

  for (int idx = tid; idx < kq * kSub; idx += blockDim.x) {
    const int j = idx / kSub, row = idx - j * kSub, s = s_begin + j * kSub + row;
    kpos[idx] = j < n_sub && s < s_end ? p.ring_pos[(size_t)seq * p.window + s] : -1;
  }
  pdl_wait();   // q and the block's keys come from the q/k/v kernel
  // independent loads: this warp's q rows, the block's keys (split 0)
  float2 qraw[HD / 16][4];
  {
    const float* qr0 = p.q + (size_t)(seq * kBlock + g) * qd + (head0 + hl) * HD;
    const float* qr1 = qr0 + (size_t)8 * qd;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const int k0 = ks * 16 + 2 * t;
      qraw[ks][0] = *reinterpret_cast<const float2*>(qr0 + k0);
      qraw[ks][1] = *reinterpret_cast<const float2*>(qr1 + k0);
      qraw[ks][2] = *reinterpret_cast<const float2*>(qr0 + k0 + 8);
      qraw[ks][3] = *reinterpret_cast<const float2*>(qr1 + k0 + 8);
    }
  }
  if (split == 0) {  // the block's own 16 keys (fp32: split hi/lo), <= 4 float4 per thread a pass
    constexpr int kBlkPer = 4, n = kBlock * (HD / 4);
    for (int base = 0; base < n; base += kBlkPer * (int)blockDim.x) {
      float4 kr[kBlkPer], vr[kBlkPer];
#pragma unroll
      for (int u = 0; u < kBlkPer; ++u) {
        const int idx = base + u * (int)blockDim.x + tid;
        kr[u] = vr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < n) {
          const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
          const size_t o = (size_t)(seq * kBlock + row) * kvd + kvh * HD + d;
          kr[u] = *reinterpret_cast<const float4*>(p.kblk + o);
          vr[u] = *reinterpret_cast<const float4*>(p.vblk + o);
        }
      }
#pragma unroll
      for (int u = 0; u < kBlkPer; ++u) {
        const int idx = base + u * (int)blockDim.x + tid;
        if (idx >= n) continue;
        const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
        uint2 h, l;
        split_bf16x2(kr[u].x, kr[u].y, h.x, l.x);
        split_bf16x2(kr[u].z, kr[u].w, h.y, l.y);
        *reinterpret_cast<uint2*>(blk_k_hi + row * KS + d) = h;
        *reinterpret_cast<uint2*>(blk_k_lo + row * KS + d) = l;
        split_bf16x2(vr[u].x, vr[u].y, h.x, l.x);
        split_bf16x2(vr[u].z, vr[u].w, h.y, l.y);
        *reinterpret_cast<uint2*>(blk_v_hi + row * KS + d) = h;
        *reinterpret_cast<uint2*>(blk_v_lo + row * KS + d) = l;
      }
    }
  }
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
  const float qscale = p.scale * kLog2e;
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      split_bf16x2(qraw[ks][e].x * qscale, qraw[ks][e].y * qscale, qh[ks][e], ql[ks][e]);
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float O[HD / 8][4];
#pragma unroll
  for (int jd = 0; jd < HD / 8; ++jd) O[jd][0] = O[jd][1] = O[jd][2] = O[jd][3] = 0.f;
  __syncthreads();  // zero-filled rows, fp32 tiles, block keys and slot positions
  if (split == 0 && lk == n_sub % kq)
    attend_tile<HD, true>(qh, ql, blk_k_hi, blk_k_lo, blk_v_hi, blk_v_lo, KS, 2, nullptr, true, p0,
                          p.window, p.block_width, m0, m1, l0, l1, O, lane);
  if (lk < n_sub) {
    if (!RING_F32 && !mbar_wait(&s_bar[lk], 0)) {
      if (lane == 0) atomicOr(p.status, 0x4u);
      mbar_wait(&s_bar[lk], 0);  // a second bounded wait before moving on
    }
    // row 0 has the widest window: a sub-chunk with no key for it has none for any row
    const int* kp = kpos + lk * kSub;
    const int ka = kp[lane], kb = kp[lane + 32];
    const bool any = __any_sync(0xffffffffu, (ka >= 0 && ka < p0 && p0 - ka < p.window) ||
                                                 (kb >= 0 && kb < p0 && p0 - kb < p.window));
    if (any) {
      const uint16_t* kh = bufs + lk * buf_elems;
      if (TMA)
        attend_tile<HD, false, true>(qh, ql, kh, nullptr, kh + SM::TILE_SW, nullptr, KS, 8, kp, false,
                                     p0, p.window, 16, m0, m1, l0, l1, O, lane);
      else
        attend_tile<HD, RING_F32>(qh, ql, kh, kh + 2 * SM::TILE, kh + SM::TILE, kh + 3 * SM::TILE, KS,
                                  8, kp, false, p0, p.window, 16, m0, m1, l0, l1, O, lane);
    }
  }
  __syncthreads();  // the staging buffers become the key-lane merge area
  // this CTA reads nothing more from HBM: its share of the next projection's
  // weights moves into L2 during the publication, group wait and merge
  if (tid == 0)
    prefetch_share_attn(p, ((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x,
                        (long long)gridDim.x * gridDim.y * gridDim.z);

  // key lanes 1.. hand their (max, sum, O) fragments to key lane 0 through
  // shared memory; it merges them in lane order and publishes the CTA's rows
  float4* frag_o = reinterpret_cast<float4*>(sm_raw);                 // [warps][HD/8][32]
  float4* frag_ml = frag_o + (size_t)nwarps * (HD / 8) * 32;          // [warps][32]
  if (lk > 0) {
#pragma unroll
    for (int jd = 0; jd < HD / 8; ++jd)
      frag_o[((size_t)warp * (HD / 8) + jd) * 32 + lane] = make_float4(O[jd][0], O[jd][1], O[jd][2], O[jd][3]);
    frag_ml[warp * 32 + lane] = make_float4(m0, m1, l0, l1);
  }
  __syncthreads();
  const size_t part0 = ((size_t)group * n_split + split) * R;   // this CTA's first partial row
  if (lk == 0) {
    for (int q = 1; q < kq; ++q) {
      const int w = warp + q;
      const float4 ml = frag_ml[w * 32 + lane];
      const float n0 = fmaxf(m0, ml.x), n1 = fmaxf(m1, ml.y);
      const float a0 = m0 == -CUDART_INF_F ? 0.f : exp2f(m0 - n0);
      const float b0 = ml.x == -CUDART_INF_F ? 0.f : exp2f(ml.x - n0);
      const float a1 = m1 == -CUDART_INF_F ? 0.f : exp2f(m1 - n1);
      const float b1 = ml.y == -CUDART_INF_F ? 0.f : exp2f(ml.y - n1);
      m0 = n0;
      m1 = n1;
      l0 = a0 * l0 + b0 * ml.z;
      l1 = a1 * l1 + b1 * ml.w;
#pragma unroll
      for (int jd = 0; jd < HD / 8; ++jd) {
        const float4 v = frag_o[((size_t)w * (HD / 8) + jd) * 32 + lane];
        O[jd][0] = a0 * O[jd][0] + b0 * v.x;
        O[jd][1] = a0 * O[jd][1] + b0 * v.y;
        O[jd][2] = a1 * O[jd][2] + b1 * v.z;
        O[jd][3] = a1 * O[jd][3] + b1 * v.w;
      }
    }
    float* o0 = p.part_o + (part0 + hl * kBlock + g) * HD;
    float* o1 = o0 + (size_t)8 * HD;
#pragma unroll
    for (int jd = 0; jd < HD / 8; ++jd) {
      __stcg(reinterpret_cast<float2*>(o0 + 8 * jd + 2 * t), make_float2(O[jd][0], O[jd][1]));
      __stcg(reinterpret_cast<float2*>(o1 + 8 * jd + 2 * t), make_float2(O[jd][2], O[jd][3]));
    }
    if (t == 0) {
      __stcg(p.part_ml + part0 + hl * kBlock + g, make_float2(m0, l0));
      __stcg(p.part_ml + part0 + hl * kBlock + g + 8, make_float2(m1, l1));
    }
  }
  // arrive (release: every thread's partial stores are ordered before it by the
  // barrier), then wait until the group's n_split CTAs have arrived (acquire)
  __syncthreads();
  int* arrive = p.counters + 2 * group;
  if (tid == 0) {
    atom_add_release_gpu(arrive, 1);
    const long long t0 = clock64();
    while (ld_acquire_gpu(arrive) < n_split) {
      if (clock64() - t0 > 4000000000LL) {
        atomicOr(p.status, 0x4u);
        break;
      }
    }
  }
  __syncthreads();

  // merge rows split, split + n_split, ... of the group: one warp per row, lane
  // c holds split c's (m, l), every lane four output dims
  for (int r = split + warp * n_split; r < R; r += nwarps * n_split) {
    const size_t row0 = (size_t)group * n_split * R + r;           // split 0's copy of row r
    float2 ml = make_float2(-CUDART_INF_F, 0.f);
    if (lane < n_split) ml = __ldcg(p.part_ml + row0 + (size_t)lane * R);
    const int d = lane * 4;
    // the first kB splits' partial rows load together with (m, l): they do not
    // depend on the weights, so the merge waits one L2 round trip, not three
    constexpr int kB = 16;
    float4 v[kB];
    auto load_rows = [&](int c0) {
#pragma unroll
      for (int u = 0; u < kB; ++u)
        v[u] = c0 + u < n_split && d < HD
                   ? __ldcg(reinterpret_cast<const float4*>(p.part_o + (row0 + (size_t)(c0 + u) * R) * HD + d))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    load_rows(0);
    const float M = warp_max(ml.x);
    const float wgt = ml.x == -CUDART_INF_F ? 0.f : exp2f(ml.x - M);
    const float L = warp_sum(wgt * ml.y);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < n_split; c0 += kB) {
      if (c0 > 0) load_rows(c0);
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const float wc = __shfl_sync(0xffffffffu, wgt, (c0 + u) & 31);   // splits in order
        if (c0 + u < n_split) {
          acc.x += wc * v[u].x;
          acc.y += wc * v[u].y;
          acc.z += wc * v[u].z;
          acc.w += wc * v[u].w;
        }
      }
    }
    if (d < HD) {
      const int h = r / kBlock, i = r - h * kBlock;
      const float inv = 1.f / L;
      const size_t at = (size_t)(seq * kBlock + i) * qd + (head0 + h) * HD + d;
      uint2 hi, lo;
      split_pair16x2(acc.x * inv, acc.y * inv, p.pair_f16 != 0, hi.x, lo.x);
      split_pair16x2(acc.z * inv, acc.w * inv, p.pair_f16 != 0, hi.y, lo.y);
      *reinterpret_cast<uint2*>(p.out_hi + at) = hi;
      *reinterpret_cast<uint2*>(p.out_lo + at) = lo;
    }
  }
  // the group's last CTA past its merge resets both counters for the next launch
  __syncthreads();
  if (tid == 0) {
    s_last = atom_add_acq_rel_gpu(arrive + 1, 1) == n_split - 1;
    if (s_last) {
      arrive[0] = 0;
      arrive[1] = 0;
    }
    stamp_finish(p.stamp);
  }
}

// ---------------------------------------------------------------------------
// Stream-K attention (batches whose split grid does not fit one wave).
//
// A planning kernel, once per step, lists every sequence's 64-slot
// sub-chunks that hold a key of block row 0's window (the widest of the
// block's rows: a sub-chunk without one has none for any row), in ring order;
// the attention CTAs sum the units per sequence into a prefix in shared memory.
// Work units are pairs of listed sub-chunks (one per key lane), at least one
// per (sequence, kv head, head group) for the block's own keys; the units of
// all groups form one axis, and a persistent grid of one CTA per SM takes
// equal contiguous ranges of it, so every CTA attends the same number of
// sub-chunks and no empty one is loaded.  One thread issues the next unit's
// copies (the ring tiles by TMA, their slot positions by a bulk copy, on one
// mbarrier per buffer set) into the other of two buffer sets while the CTA
// attends the current one.  A group wholly inside one CTA's range is
// normalised and written at once; a group cut by range boundaries publishes
// one partial per contributor (slot 2c for the part that starts CTA c's range
// or lies inside it, 2c + 1 for the part that ends it) and the last
// contributor (acquire-release ticket) merges them in CTA order, so results do
// not depend on timing.  The block's own keys are attended with the group's
// first unit.
// ---------------------------------------------------------------------------

constexpr int kStreamKq = 2;       // key lanes (sub-chunks per unit)
constexpr int kStreamMaxSub = 64;  // 64-slot sub-chunks per window (window <= 4096)

// One CTA per sequence, one thread per 64-slot sub-chunk (window <= 4096): all
// of a sub-chunk's 64 slot positions are loaded at once.
__global__ void __launch_bounds__(kStreamMaxSub) attn_plan_kernel(const int32_t* ring_pos, const int32_t* n_past,
                                                                  int window, int* nv, int* sub) {
  const int s = blockIdx.x, sc = threadIdx.x, lane = sc & 31, w = sc >> 5;
  const int n_sub = (window + kSub - 1) / kSub;
  const int p0 = max(n_past[s], 0);
  bool any = false;
  if (sc < n_sub) {
    const int s0 = sc * kSub, nk4 = min(kSub, window - s0) / 4;   // the window is a multiple of 4 slots
    const int4* rp = reinterpret_cast<const int4*>(ring_pos + (size_t)s * window + s0);
    int4 k4[kSub / 4];
#pragma unroll
    for (int i = 0; i < kSub / 4; ++i) k4[i] = i < nk4 ? __ldg(rp + i) : make_int4(-1, -1, -1, -1);
#pragma unroll
    for (int i = 0; i < kSub / 4; ++i) {
      const int kk[4] = {k4[i].x, k4[i].y, k4[i].z, k4[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) any |= kk[q] >= 0 && kk[q] < p0 && p0 - kk[q] < window;
    }
  }
  __shared__ unsigned s_ball[kStreamMaxSub / 32];
  const unsigned bal = __ballot_sync(0xffffffffu, any);
  if (lane == 0) s_ball[w] = bal;
  __syncthreads();
  int before = __popc(bal & ((1u << lane) - 1u)), total = 0;
  for (int i = 0; i < kStreamMaxSub / 32; ++i) {
    if (i < w) before += __popc(s_ball[i]);
    total += __popc(s_ball[i]);
  }
  if (any) sub[(size_t)s * kStreamMaxSub + before] = sc;
  if (sc == 0) nv[s] = total;
}

template <int HD>
struct StreamSmem {
  using SM = AttnSmem<HD>;
  static constexpr size_t SET = (size_t)kStreamKq * 2 * SM::TILE_SW * 2;   // K + V tiles of each lane
  static constexpr size_t OFF_BLK = 2 * SET;
  static constexpr size_t OFF_FRAG = OFF_BLK + (size_t)SM::BLK * 2;
  static constexpr size_t OFF_KPOS = OFF_FRAG + (size_t)4 * (HD / 8) * 32 * 16 + (size_t)4 * 32 * 16;
  static constexpr size_t OFF_PLAN = OFF_KPOS + (size_t)2 * kStreamKq * kSub * 4;
  static constexpr size_t BYTES = OFF_PLAN + (size_t)(2 * kAttnStreamMaxSeq + 1) * 4 + 1024;   // + alignment
};

template <int HD>
__global__ void __launch_bounds__(256, 1) attn_stream_kernel(const __grid_constant__ AttnParams p) {
  using SM = AttnSmem<HD>;
  using SS = StreamSmem<HD>;
  constexpr int KS = SM::KS, TS = SM::TILE_SW, KQ = kStreamKq;
  const int G = p.n_head / p.n_head_kv, hpc = p.hpc, n_hgrp = G / hpc;
  const int gps = p.n_head_kv * n_hgrp;   // groups per sequence
  const int qd = p.n_head * HD, kvd = p.n_head_kv * HD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int nthreads = (int)blockDim.x;
  const int hl = warp / KQ, lk = warp - hl * KQ;
  const int R = kBlock * hpc;
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint16_t* sets = reinterpret_cast<uint16_t*>(base);   // [2][KQ][K tile, V tile]
  uint16_t* blk_k_hi = reinterpret_cast<uint16_t*>(base + SS::OFF_BLK);
  uint16_t* blk_k_lo = blk_k_hi + kBlock * KS;
  uint16_t* blk_v_hi = blk_k_lo + kBlock * KS;
  uint16_t* blk_v_lo = blk_v_hi + kBlock * KS;
  float4* frag_o = reinterpret_cast<float4*>(base + SS::OFF_FRAG);   // key lane 1: [hpc][HD/8][32]
  float4* frag_ml = frag_o + (size_t)4 * (HD / 8) * 32;               // [hpc][32]
  int* kpos = reinterpret_cast<int*>(base + SS::OFF_KPOS);            // [2][KQ][64]
  int* s_prefix = reinterpret_cast<int*>(base + SS::OFF_PLAN);        // [n_seq + 1] units before each sequence
  int* s_nv = s_prefix + p.n_seq + 1;                                 // [n_seq] listed sub-chunks
  __shared__ __align__(8) uint64_t s_bar[2];
  __shared__ int s_flag;

  // the plan was written by the kernel before the step's first projection
  // (which starts only once the plan kernel has completed): units of each
  // sequence -> exclusive prefix over sequences (a block scan)
  __shared__ int s_wsum[8];
  {
    const int per = (p.n_seq + nthreads - 1) / nthreads;
    const int i0 = min(p.n_seq, tid * per), i1 = min(p.n_seq, i0 + per);
    int local = 0;
    for (int i = i0; i < i1; ++i) {
      const int v = p.plan_nv[i];
      s_nv[i] = v;
      local += max(1, (v + 1) / 2) * gps;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += s_wsum[w];
    for (int i = i0; i < i1; ++i) {
      s_prefix[i] = run;
      run += max(1, (s_nv[i] + 1) / 2) * gps;
    }
    if (tid == nthreads - 1) s_prefix[p.n_seq] = run;
  }
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    stamp_begin(p.stamp);
  }
  __syncthreads();
  pdl_trigger();
  const long long T = s_prefix[p.n_seq];
  const int b = blockIdx.x, GC = gridDim.x;
  const long long u0 = T * b / GC, u1 = T * (b + 1) / GC;
  auto owner = [&](long long u) { return (int)(((u + 1) * GC - 1) / T); };
  const size_t plane = (size_t)p.window * HD;
  struct Unit {
    int seq, gi, k, nu, nv;
  };
  auto decode = [&](long long u) {
    int lo = 0, hi = p.n_seq;   // the sequence s with prefix[s] <= u < prefix[s + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_prefix[mid] <= u) lo = mid; else hi = mid;
    }
    Unit x;
    x.seq = lo;
    x.nv = s_nv[lo];
    x.nu = max(1, (x.nv + 1) / 2);
    const int local = (int)(u - s_prefix[lo]);
    x.gi = local / x.nu;
    x.k = local - x.gi * x.nu;
    return x;
  };

  // copies of unit u into buffer set st (thread 0): the unit's listed
  // sub-chunks (zero-filled past the tensor; a slot past the window gets
  // position -1)
  auto issue = [&](long long u, int st) {
    const Unit x = decode(u);
    const int kvh = x.gi / n_hgrp;
    const size_t kbase = ((((size_t)x.seq * p.n_layer + p.layer) * 2 + 0) * p.n_head_kv + kvh) * plane;
    const int row_k = (int)(kbase / HD), row_v = (int)((kbase + (size_t)p.n_head_kv * plane) / HD);
    uint32_t bytes = 0;
    int s0s[KQ], nks[KQ];
#pragma unroll
    for (int j = 0; j < KQ; ++j) {
      const int li = 2 * x.k + j;
      s0s[j] = li < x.nv ? p.plan_sub[(size_t)x.seq * kStreamMaxSub + li] * kSub : p.window;
      nks[j] = s0s[j] < p.window ? min(kSub, p.window - s0s[j]) : 0;
      if (nks[j] > 0) bytes += (uint32_t)(2 * TS * 2 + nks[j] * 4);
    }
    mbar_expect_tx(&s_bar[st], bytes);
#pragma unroll
    for (int j = 0; j < KQ; ++j) {
      int* kp = kpos + (st * KQ + j) * kSub;
      for (int i = nks[j]; i < kSub; ++i) kp[i] = -1;
      if (nks[j] == 0) continue;
      uint16_t* dst = sets + ((size_t)st * KQ + j) * 2 * TS;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv)
#pragma unroll
        for (int hb = 0; hb < HD / 64; ++hb)
          tma_load_2d(dst + kv * TS + hb * kSub * 64, &p.tm_ring, hb * 64, (kv ? row_v : row_k) + s0s[j],
                      &s_bar[st]);
      bulk_copy(kp, p.ring_pos + (size_t)x.seq * p.window + s0s[j], (uint32_t)nks[j] * 4, &s_bar[st]);
    }
  };

  // the ring and its slot positions were written before the step's first
  // kernel (launched without overlap): the first unit is staged before the
  // wait for the q/k/v kernel
  if (tid == 0 && u0 < u1) issue(u0, 0);
  pdl_wait();

  const float qscale = p.scale * kLog2e;
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float O[HD / 8][4];
  for (long long u = u0; u < u1; ++u) {
    const int it = (int)(u - u0), st = it & 1;
    __syncthreads();   // unit it - 1 is done with the other set, the block keys and the merge area
    if (tid == 0 && u + 1 < u1) issue(u + 1, st ^ 1);
    const Unit x = decode(u);
    const int seq = x.seq, kvh = x.gi / n_hgrp, hg = x.gi - kvh * n_hgrp;
    const int group = seq * gps + x.gi;
    const int head0 = kvh * G + hg * hpc;
    const int p0 = max(p.n_past[seq], 0);
    const bool seg_first = u == u0 || x.k == 0, seg_last = u + 1 == u1 || x.k == x.nu - 1;
    if (seg_first) {
      const float* qr0 = p.q + (size_t)(seq * kBlock + g) * qd + (head0 + hl) * HD;
      const float* qr1 = qr0 + (size_t)8 * qd;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        const int k0 = ks * 16 + 2 * t;
        const float2 a0 = *reinterpret_cast<const float2*>(qr0 + k0);
        const float2 a1 = *reinterpret_cast<const float2*>(qr1 + k0);
        const float2 a2 = *reinterpret_cast<const float2*>(qr0 + k0 + 8);
        const float2 a3 = *reinterpret_cast<const float2*>(qr1 + k0 + 8);
        split_bf16x2(a0.x * qscale, a0.y * qscale, qh[ks][0], ql[ks][0]);
        split_bf16x2(a1.x * qscale, a1.y * qscale, qh[ks][1], ql[ks][1]);
        split_bf16x2(a2.x * qscale, a2.y * qscale, qh[ks][2], ql[ks][2]);
        split_bf16x2(a3.x * qscale, a3.y * qscale, qh[ks][3], ql[ks][3]);
      }
      m0 = m1 = -CUDART_INF_F;
      l0 = l1 = 0.f;
#pragma unroll
      for (int jd = 0; jd < HD / 8; ++jd) O[jd][0] = O[jd][1] = O[jd][2] = O[jd][3] = 0.f;
    }
    if (x.k == 0) {   // the group's first unit: the block's own 16 keys
      for (int idx = tid; idx < kBlock * (HD / 4); idx += nthreads) {
        const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
        const size_t o = (size_t)(seq * kBlock + row) * kvd + kvh * HD + d;
        const float4 kr = *reinterpret_cast<const float4*>(p.kblk + o);
        const float4 vr = *reinterpret_cast<const float4*>(p.vblk + o);
        uint2 h, l;
        split_bf16x2(kr.x, kr.y, h.x, l.x);
        split_bf16x2(kr.z, kr.w, h.y, l.y);
        *reinterpret_cast<uint2*>(blk_k_hi + row * KS + d) = h;
        *reinterpret_cast<uint2*>(blk_k_lo + row * KS + d) = l;
        split_bf16x2(vr.x, vr.y, h.x, l.x);
        split_bf16x2(vr.z, vr.w, h.y, l.y);
        *reinterpret_cast<uint2*>(blk_v_hi + row * KS + d) = h;
        *reinterpret_cast<uint2*>(blk_v_lo + row * KS + d) = l;
      }
      __syncthreads();
      // the lane without a listed sub-chunk when the group has an odd count
      if (lk == KQ - 1)
        attend_tile<HD, true>(qh, ql, blk_k_hi, blk_k_lo, blk_v_hi, blk_v_lo, KS, 2, nullptr, true, p0,
                              p.window, p.block_width, m0, m1, l0, l1, O, lane);
    }
    if (!mbar_wait(&s_bar[st], (uint32_t)((it >> 1) & 1))) {
      if (lane == 0) atomicOr(p.status, 0x4u);
      mbar_wait(&s_bar[st], (uint32_t)((it >> 1) & 1));   // a second bounded wait before moving on
    }
    if (2 * x.k + lk < x.nv) {
      const int* kp = kpos + (st * KQ + lk) * kSub;
      const uint16_t* kh = sets + ((size_t)st * KQ + lk) * 2 * TS;
      attend_tile<HD, false, true>(qh, ql, kh, nullptr, kh + TS, nullptr, KS, 8, kp, false, p0, p.window, 16,
                                   m0, m1, l0, l1, O, lane);
    }
    if (!seg_last) continue;

    // ---- the segment's last unit: merge the key lanes (lane order), then
    // write the group's output or this contributor's partial
    if (lk > 0) {
#pragma unroll
      for (int jd = 0; jd < HD / 8; ++jd)
        frag_o[((size_t)hl * (HD / 8) + jd) * 32 + lane] = make_float4(O[jd][0], O[jd][1], O[jd][2], O[jd][3]);
      frag_ml[hl * 32 + lane] = make_float4(m0, m1, l0, l1);
    }
    __syncthreads();
    if (lk == 0) {
      const float4 ml = frag_ml[hl * 32 + lane];
      const float n0 = fmaxf(m0, ml.x), n1 = fmaxf(m1, ml.y);
      const float a0 = m0 == -CUDART_INF_F ? 0.f : exp2f(m0 - n0);
      const float b0 = ml.x == -CUDART_INF_F ? 0.f : exp2f(ml.x - n0);
      const float a1 = m1 == -CUDART_INF_F ? 0.f : exp2f(m1 - n1);
      const float b1 = ml.y == -CUDART_INF_F ? 0.f : exp2f(ml.y - n1);
      m0 = n0;
      m1 = n1;
      l0 = a0 * l0 + b0 * ml.z;
      l1 = a1 * l1 + b1 * ml.w;
#pragma unroll
      for (int jd = 0; jd < HD / 8; ++jd) {
        const float4 v = frag_o[((size_t)hl * (HD / 8) + jd) * 32 + lane];
        O[jd][0] = a0 * O[jd][0] + b0 * v.x;
        O[jd][1] = a0 * O[jd][1] + b0 * v.y;
        O[jd][2] = a1 * O[jd][2] + b1 * v.z;
        O[jd][3] = a1 * O[jd][3] + b1 * v.w;
      }
    }
    const long long gu0 = s_prefix[seq] + (long long)x.gi * x.nu;
    const int first = owner(gu0), last = owner(gu0 + x.nu - 1);
    if (first == last) {   // the whole window in this CTA: normalise and write
      if (lk == 0) {
        const float i0 = 1.f / l0, i1 = 1.f / l1;
        uint16_t* oh = p.out_hi + (size_t)(seq * kBlock + g) * qd + (head0 + hl) * HD + 2 * t;
        uint16_t* ol = p.out_lo + (size_t)(seq * kBlock + g) * qd + (head0 + hl) * HD + 2 * t;
#pragma unroll
        for (int jd = 0; jd < HD / 8; ++jd) {
          uint32_t h, l;
          split_pair16x2(O[jd][0] * i0, O[jd][1] * i0, p.pair_f16 != 0, h, l);
          *reinterpret_cast<uint32_t*>(oh + 8 * jd) = h;
          *reinterpret_cast<uint32_t*>(ol + 8 * jd) = l;
          split_pair16x2(O[jd][2] * i1, O[jd][3] * i1, p.pair_f16 != 0, h, l);
          *reinterpret_cast<uint32_t*>(oh + (size_t)8 * qd + 8 * jd) = h;
          *reinterpret_cast<uint32_t*>(ol + (size_t)8 * qd + 8 * jd) = l;
        }
      }
      continue;
    }
    auto slot_of = [&](int c) { return (size_t)(2 * c + (c == first ? 1 : 0)) * R; };
    if (lk == 0) {
      const size_t row0 = slot_of(b) + hl * kBlock + g;
      float* o0 = p.part_o + row0 * HD + 2 * t;
      float* o1 = o0 + (size_t)8 * HD;
#pragma unroll
      for (int jd = 0; jd < HD / 8; ++jd) {
        __stcg(reinterpret_cast<float2*>(o0 + 8 * jd), make_float2(O[jd][0], O[jd][1]));
        __stcg(reinterpret_cast<float2*>(o1 + 8 * jd), make_float2(O[jd][2], O[jd][3]));
      }
      if (t == 0) {
        __stcg(p.part_ml + row0, make_float2(m0, l0));
        __stcg(p.part_ml + row0 + 8, make_float2(m1, l1));
      }
    }
    // ticket (acquire-release; the barrier orders every thread's partial
    // stores before it): the last contributor merges the group
    __syncthreads();
    if (tid == 0) {
      int* cnt = p.counters + 2 * group;
      s_flag = atom_add_acq_rel_gpu(cnt, 1) == last - first;
      if (s_flag) *cnt = 0;
    }
    __syncthreads();
    if (!s_flag) continue;
    // merge: thread -> (row, 4 dims); contributors in CTA order, online rescale
    constexpr int kB = 4;
    for (int i0 = tid; i0 < R * (HD / 4); i0 += kB * nthreads) {
      float M[kB], L[kB];
      float4 acc[kB];
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        M[q] = -CUDART_INF_F;
        L[q] = 0.f;
        acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int c = first; c <= last; ++c) {
        const size_t s0 = slot_of(c);
        float2 ml[kB];
        float4 v[kB];
#pragma unroll
        for (int q = 0; q < kB; ++q) {
          const int idx = i0 + q * nthreads;
          if (idx < R * (HD / 4)) {
            const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
            ml[q] = __ldcg(p.part_ml + s0 + row);
            v[q] = __ldcg(reinterpret_cast<const float4*>(p.part_o + (s0 + row) * HD + d));
          }
        }
#pragma unroll
        for (int q = 0; q < kB; ++q) {
          if (i0 + q * nthreads >= R * (HD / 4)) continue;
          const float n = fmaxf(M[q], ml[q].x);
          const float a = M[q] == -CUDART_INF_F ? 0.f : exp2f(M[q] - n);
          const float w = ml[q].x == -CUDART_INF_F ? 0.f : exp2f(ml[q].x - n);
          M[q] = n;
          L[q] = a * L[q] + w * ml[q].y;
          acc[q].x = a * acc[q].x + w * v[q].x;
          acc[q].y = a * acc[q].y + w * v[q].y;
          acc[q].z = a * acc[q].z + w * v[q].z;
          acc[q].w = a * acc[q].w + w * v[q].w;
        }
      }
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int idx = i0 + q * nthreads;
        if (idx >= R * (HD / 4)) continue;
        const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
        const int h = row / kBlock, i = row - h * kBlock;
        const float inv = 1.f / L[q];
        const size_t at = (size_t)(seq * kBlock + i) * qd + (head0 + h) * HD + d;
        uint2 hi, lo;
        split_pair16x2(acc[q].x * inv, acc[q].y * inv, p.pair_f16 != 0, hi.x, lo.x);
        split_pair16x2(acc[q].z * inv, acc[q].w * inv, p.pair_f16 != 0, hi.y, lo.y);
        *reinterpret_cast<uint2*>(p.out_hi + at) = hi;
        *reinterpret_cast<uint2*>(p.out_lo + at) = lo;
      }
    }
  }
  __syncthreads();
  if (tid == 0) stamp_finish(p.stamp);
}

int attn_cluster_size(int window) {
  int cl = (window + 255) / 256;
  return cl < 1 ? 1 : (cl > kMaxCluster ? kMaxCluster : cl);
}

template <int HD>
static size_t smem_of(bool f32, const AttnPlan& pl) {
  return AttnSmem<HD>::bytes(f32, pl);
}
static size_t smem_of_hd(int hd, bool f32, const AttnPlan& pl) {
  switch (hd) {
    case 32: return smem_of<32>(f32, pl);
    case 64: return smem_of<64>(f32, pl);
    default: return smem_of<128>(f32, pl);
  }
}

size_t attn_cluster_smem(int group, int hd, int ring_f32) {
  AttnPlan pls[kLatencyPlans + 1];
  const int n = plans_for(ring_f32 != 0, group, 1 << 20, pls);   // the deepest staging of any window
  size_t best = 0;
  for (int i = 0; i < n; ++i) {
    const size_t b = smem_of_hd(hd, ring_f32 != 0, pls[i]);
    if (b > best) best = b;
  }
  return best;
}

// Co-resident clusters of each plan, measured with the occupancy API once per
// (kernel, plan, cluster size) when a handle is created, so that launches
// (also under stream capture) only read the table.
struct OccEntry {
  const void* fn;
  int threads, cl;
  size_t smem;
  int clusters;
};
static std::mutex g_occ_mu;
static std::vector<OccEntry> g_occ;

template <int HD, bool F32>
static int active_clusters(const AttnPlan& pl, int CL, bool query) {
  const void* fn = reinterpret_cast<const void*>(attn_cluster_kernel<HD, F32>);
  const int threads = 32 * pl.hpc * pl.kq;
  const size_t smem = smem_of<HD>(F32, pl);
  std::lock_guard<std::mutex> lk(g_occ_mu);
  for (const OccEntry& e : g_occ)
    if (e.fn == fn && e.threads == threads && e.cl == CL && e.smem == smem) return e.clusters;
  if (!query) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, 1, 1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_cluster_kernel<HD, F32>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  g_occ.push_back(OccEntry{fn, threads, CL, smem, n});
  return n;
}

// The plan of a launch: the latency plan with the least estimated time when
// the grid fits in a few waves of co-resident clusters, else the throughput
// plan.  Estimated time = waves x (1 + tiles per warp x warps per SM
// sub-partition), in units of one tile.
template <int HD, bool F32>
static AttnPlan choose_plan(int G, int CL, int n_head_kv, int n_seq, int window, bool query) {
  AttnPlan pls[kLatencyPlans + 1];
  const int per = (window + CL - 1) / CL, n_sub = (per + kSub - 1) / kSub;
  const int n = plans_for(F32, G, n_sub, pls);
  AttnPlan best = pls[n - 1];
  double best_cost = 1e30;
  for (int i = 0; i < n - 1; ++i) {
    const AttnPlan& pl = pls[i];
    const int act = active_clusters<HD, F32>(pl, CL, query);
    if (act <= 0) continue;
    const long long clusters = (long long)n_head_kv * (G / pl.hpc) * n_seq;
    const long long waves = (clusters + act - 1) / act;
    if (waves > 2) continue;
    const int tiles = (n_sub + pl.kq - 1) / pl.kq;
    const int per_smsp = (pl.hpc * pl.kq + 3) / 4;
    const double cost = (double)waves * (1.0 + (double)tiles * per_smsp);
    if (cost < best_cost) {
      best_cost = cost;
      best = pl;
    }
  }
  return best;
}

template <int HD, bool F32>
static cudaError_t configure_cl(size_t smem, int G, int CL, int n_head_kv, int window) {
  static size_t configured = 0;   // only ever raised, so every live handle still fits
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<HD, F32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  AttnPlan pls[kLatencyPlans + 1];
  const int per = (window + CL - 1) / CL, n_sub = (per + kSub - 1) / kSub;
  const int n = plans_for(F32, G, n_sub, pls);
  for (int i = 0; i < n; ++i) (void)active_clusters<HD, F32>(pls[i], CL, true);
  (void)n_head_kv;
  return cudaSuccess;
}

cudaError_t configure_attention_cluster(int group, int hd, int ring_f32, int window, int n_head_kv) {
  const size_t smem = attn_cluster_smem(group, hd, ring_f32);
  const int CL = attn_cluster_size(window);
  switch (hd) {
    case 32: return ring_f32 ? configure_cl<32, true>(smem, group, CL, n_head_kv, window)
                             : configure_cl<32, false>(smem, group, CL, n_head_kv, window);
    case 64: return ring_f32 ? configure_cl<64, true>(smem, group, CL, n_head_kv, window)
                             : configure_cl<64, false>(smem, group, CL, n_head_kv, window);
    case 128: return ring_f32 ? configure_cl<128, true>(smem, group, CL, n_head_kv, window)
                              : configure_cl<128, false>(smem, group, CL, n_head_kv, window);
  }
  return cudaErrorInvalidValue;
}

template <int HD, bool F32>
static cudaError_t launch_cl(const AttnParams& p_in, int n_seq, cudaStream_t st) {
  const int G = p_in.n_head / p_in.n_head_kv;
  int CL = attn_cluster_size(p_in.window);
  const AttnPlan pl = choose_plan<HD, F32>(G, CL, p_in.n_head_kv, n_seq, p_in.window, false);
  // a batch large enough to fill the GPU twice without splitting windows gives
  // each CTA a whole window: no cluster merge, and the prologue and merge are
  // paid once per window instead of once per slice
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (n_sm <= 0) n_sm = 1;
  }
  if ((long long)p_in.n_head_kv * (G / pl.hpc) * n_seq >= 2LL * n_sm) CL = 1;
  AttnParams p = p_in;
  p.hpc = pl.hpc;
  p.kq = pl.kq;
  p.nb = pl.nb;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, p.n_head_kv * (G / pl.hpc), n_seq);
  cfg.blockDim = dim3(32 * pl.kq * pl.hpc);
  cfg.dynamicSmemBytes = smem_of<HD>(F32, pl);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<HD, F32>, p);
}

cudaError_t launch_attention_cluster(const AttnParams& p, int n_seq, cudaStream_t st) {
  const bool f32 = !p.ring_bf16;
  switch (p.hd) {
    case 32: return f32 ? launch_cl<32, true>(p, n_seq, st) : launch_cl<32, false>(p, n_seq, st);
    case 64: return f32 ? launch_cl<64, true>(p, n_seq, st) : launch_cl<64, false>(p, n_seq, st);
    case 128: return f32 ? launch_cl<128, true>(p, n_seq, st) : launch_cl<128, false>(p, n_seq, st);
  }
  return cudaErrorInvalidValue;
}

// ---- split-window launch plan: kq = 2 key lanes (128 slots per CTA), up to 4
// query heads of the kv group per CTA
struct SplitPlan {
  int hpc, kq, n_split;
};
inline SplitPlan split_plan(int G, int window) {
  SplitPlan s;
  s.kq = 2;
  s.hpc = G % 4 == 0 ? 4 : G % 2 == 0 ? 2 : 1;
  s.n_split = (window + s.kq * kSub - 1) / (s.kq * kSub);
  return s;
}
template <int HD>
static size_t split_smem_of(bool f32, const SplitPlan& s) {
  using SM = AttnSmem<HD>;
  const size_t stage = (size_t)s.kq * SM::buf_elems(f32) * 2 + (size_t)SM::BLK * 2 +
                       (size_t)s.kq * kSub * 4 + (SM::kTma && !f32 ? 1024 : 0);
  const int warps = s.hpc * s.kq;
  const size_t merge = (size_t)warps * (HD / 8) * 32 * 16 + (size_t)warps * 32 * 16;
  return (stage > merge ? stage : merge) + 256;
}
static size_t split_smem_hd(int hd, bool f32, const SplitPlan& s) {
  switch (hd) {
    case 32: return split_smem_of<32>(f32, s);
    case 64: return split_smem_of<64>(f32, s);
    default: return split_smem_of<128>(f32, s);
  }
}
size_t attn_split_smem(int group, int hd, int ring_f32) {
  return split_smem_hd(hd, ring_f32 != 0, split_plan(group, 64));
}

// CTAs of the split kernel the GPU holds at once, measured with the occupancy
// API when a handle is created (launches, also under capture, read the table)
struct SplitCap {
  const void* fn;
  int threads;
  size_t smem;
  int ctas;
};
static std::vector<SplitCap> g_split_cap;

template <int HD, bool F32>
static int split_capacity(const SplitPlan& s, bool query) {
  const void* fn = reinterpret_cast<const void*>(attn_split_kernel<HD, F32>);
  const int threads = 32 * s.hpc * s.kq;
  const size_t smem = split_smem_of<HD>(F32, s);
  std::lock_guard<std::mutex> lk(g_occ_mu);
  for (const SplitCap& c : g_split_cap)
    if (c.fn == fn && c.threads == threads && c.smem == smem) return c.ctas;
  if (!query) return 0;
  int per_sm = 0, dev = 0, n_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_kernel<HD, F32>, threads, smem) !=
          cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    per_sm = 0;
  }
  g_split_cap.push_back(SplitCap{fn, threads, smem, per_sm * n_sm});
  return per_sm * n_sm;
}

// ---- stream-K launch: bf16 ring staged by TMA (hd >= 64), a window of at most
// kStreamMaxSub sub-chunks whose length is a multiple of 4 slots (16-byte
// copies of the slot positions), one CTA per SM
static int g_n_sm = 0;
static int sm_count() {
  if (!g_n_sm) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      g_n_sm = n;
    else
      (void)cudaGetLastError();
  }
  return g_n_sm > 0 ? g_n_sm : 1;
}
template <int HD>
static cudaError_t configure_stream() {
  static bool done = false;
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_stream_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)StreamSmem<HD>::BYTES);
  if (e == cudaSuccess) done = true;
  (void)sm_count();
  return e;
}
template <int HD, bool F32>
static bool stream_fits(const AttnParams& p, int n_seq) {
  return !F32 && HD >= 64 && p.part_o && p.plan_nv && p.window % 4 == 0 &&
         (p.window + kSub - 1) / kSub <= kStreamMaxSub && n_seq <= kAttnStreamMaxSeq;
}
template <int HD>
static cudaError_t launch_stream(const AttnParams& p_in, int n_seq, int hpc, cudaStream_t st) {
  AttnParams p = p_in;
  const int G = p.n_head / p.n_head_kv;
  p.hpc = hpc;
  p.kq = kStreamKq;
  p.nb = 2 * kStreamKq;
  p.n_seq = n_seq;
  // the units are counted on the device: one CTA per SM (those past the units
  // find an empty range); two partial slots per CTA
  const int grid = std::min(sm_count(), kAttnSplitMaxCtas / 2);
  (void)G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(32 * hpc * kStreamKq);
  cfg.dynamicSmemBytes = StreamSmem<HD>::BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_stream_kernel<HD>, p);
}

template <int HD, bool F32>
static cudaError_t configure_split(int G, int window) {
  static size_t configured = 0;   // only ever raised, so every live handle still fits
  const SplitPlan s = split_plan(G, window);
  const size_t smem = split_smem_of<HD>(F32, s);
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<HD, F32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  (void)split_capacity<HD, F32>(s, true);
  return cudaSuccess;
}

cudaError_t configure_attention(int group, int hd, int ring_f32, int window, int n_head_kv) {
  cudaError_t e = configure_attention_cluster(group, hd, ring_f32, window, n_head_kv);
  if (e != cudaSuccess) return e;
  if (!ring_f32 && hd == 64) e = configure_stream<64>();
  if (!ring_f32 && hd == 128) e = configure_stream<128>();
  if (e != cudaSuccess) return e;
  switch (hd) {
    case 32: return ring_f32 ? configure_split<32, true>(group, window) : configure_split<32, false>(group, window);
    case 64: return ring_f32 ? configure_split<64, true>(group, window) : configure_split<64, false>(group, window);
    case 128: return ring_f32 ? configure_split<128, true>(group, window) : configure_split<128, false>(group, window);
  }
  return cudaErrorInvalidValue;
}

// Which kernel a step of n_seq sequences takes: the split kernel when its grid
// is resident at once, else stream-K where it applies, else clusters.
template <int HD, bool F32>
static int attention_kind_t(const AttnParams& p, int n_seq) {
  const int G = p.n_head / p.n_head_kv;
  const SplitPlan s = split_plan(G, p.window);
  const long long grid = (long long)n_seq * p.n_head_kv * (G / s.hpc) * s.n_split;
  const int cap = split_capacity<HD, F32>(s, false);
  if (p.part_o && s.n_split <= kMaxSplit && grid <= cap && grid <= kAttnSplitMaxCtas) return ATTN_SPLIT;
  return stream_fits<HD, F32>(p, n_seq) ? ATTN_STREAM : ATTN_CLUSTER;
}

template <int HD, bool F32>
static cudaError_t launch_split_or_cluster(const AttnParams& p_in, int n_seq, cudaStream_t st) {
  const int G = p_in.n_head / p_in.n_head_kv;
  const SplitPlan s = split_plan(G, p_in.window);
  const int kind = attention_kind_t<HD, F32>(p_in, n_seq);
  if (kind == ATTN_STREAM) {
    if constexpr (!F32 && HD >= 64) return launch_stream<HD>(p_in, n_seq, s.hpc, st);
  }
  if (kind != ATTN_SPLIT) return launch_cl<HD, F32>(p_in, n_seq, st);
  AttnParams p = p_in;
  p.hpc = s.hpc;
  p.kq = s.kq;
  p.nb = s.kq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.n_split, p.n_head_kv * (G / s.hpc), n_seq);
  cfg.blockDim = dim3(32 * s.hpc * s.kq);
  cfg.dynamicSmemBytes = split_smem_of<HD>(F32, s);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_split_kernel<HD, F32>, p);
}

cudaError_t launch_attention_plan(const AttnParams& p, int n_seq, cudaStream_t st) {
  const int G = p.n_head / p.n_head_kv;
  const int hpc = split_plan(G, p.window).hpc;
  // no programmatic-launch attribute and no early trigger: the next kernel
  // starts once the plan is complete and visible
  (void)hpc;
  attn_plan_kernel<<<n_seq, kStreamMaxSub, 0, st>>>(p.ring_pos, p.n_past, p.window, p.plan_nv, p.plan_sub);
  return cudaGetLastError();
}

int attention_kind(const AttnParams& p, int n_seq) {
  const bool f32 = !p.ring_bf16;
  switch (p.hd) {
    case 32: return f32 ? attention_kind_t<32, true>(p, n_seq) : attention_kind_t<32, false>(p, n_seq);
    case 64: return f32 ? attention_kind_t<64, true>(p, n_seq) : attention_kind_t<64, false>(p, n_seq);
    case 128: return f32 ? attention_kind_t<128, true>(p, n_seq) : attention_kind_t<128, false>(p, n_seq);
  }
  return ATTN_CLUSTER;
}

cudaError_t launch_attention(const AttnParams& p, int n_seq, cudaStream_t st) {
  const bool f32 = !p.ring_bf16;
  switch (p.hd) {
    case 32: return f32 ? launch_split_or_cluster<32, true>(p, n_seq, st) : launch_split_or_cluster<32, false>(p, n_seq, st);
    case 64: return f32 ? launch_split_or_cluster<64, true>(p, n_seq, st) : launch_split_or_cluster<64, false>(p, n_seq, st);
    case 128: return f32 ? launch_split_or_cluster<128, true>(p, n_seq, st) : launch_split_or_cluster<128, false>(p, n_seq, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dflash
