// Sliding-window GQA attention of the noise block, one thread-block cluster per
// (sequence, kv head).
//
// The block's 16 rows at positions n_past .. n_past + 15 attend (non-causally)
// to every row of the block and to the ring slots holding positions p with
// 0 <= p < n_past and (n_past + i) - p < window (dflash-ops model card, Method).
// The ring of one kv head is split between the CL CTAs of a cluster; each CTA
// walks its slots in 64-key sub-chunks (double-buffered async copies of the bf16
// K/V rows) with an online softmax, one warp per query head of the kv group
// (the G heads share every K/V tile).  Both products use the tensor cores with
// fp32 accumulation: q and the probabilities are split into bf16 hi + lo, bf16
// ring K/V are exact, fp32 K/V (an fp32 ring, the block's own keys) are split
// too.  The CTAs then merge their (max, sum, O) partials through distributed
// shared memory in rank order and write the o projection's input as a bf16
// hi/lo pair.  Rank 0 also attends to the block's own keys.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

#include <math_constants.h>

namespace cg = cooperative_groups;

namespace dflash {

constexpr int kSub = 64;       // keys per sub-chunk
constexpr int kPad = 8;        // bf16 row padding (conflict-free fragment loads)
constexpr int kMaxCluster = 8;

DF_DEVICE void cp16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
DF_DEVICE void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DF_DEVICE void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

DF_DEVICE void ldsm_x4_t(uint32_t (&r)[4], const void* smem) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

// Ring sub-chunks in flight per CTA.  A bf16 ring keeps four in flight when the
// grid is at most one CTA per SM (latency-bound single sequences) and two when
// it is larger, so that two CTAs fit one SM; an fp32 ring's hi/lo tiles take
// twice the room and always use two.
constexpr int kMaxDepth = 4;
inline int depth_for(bool f32, long long ctas, int n_sm) {
  return f32 || ctas > n_sm ? 2 : kMaxDepth;
}

template <int HD>
struct AttnSmem {
  static constexpr int KS = HD + kPad;
  static constexpr int TILE = kSub * KS;               // one [64][KS] bf16 tile (elements)
  // buffer b: K hi, V hi, K lo, V lo (lo only used by an fp32 ring)
  static constexpr int BUF = 4 * TILE;
  static constexpr int BLK = 4 * kBlock * KS;          // block keys: K hi/lo, V hi/lo [16][KS]
  static size_t bytes(bool f32, int depth) {
    const size_t bufs = depth * (size_t)(f32 ? BUF : 2 * TILE) * 2;
    return bufs + (size_t)BLK * 2 + kMaxDepth * kSub * sizeof(int) + 256;
  }
};

DF_DEVICE void cp_wait_upto(int n) {
  switch (n) {
    case 0: cp_wait<0>(); break;
    case 1: cp_wait<1>(); break;
    case 2: cp_wait<2>(); break;
    default: cp_wait<3>(); break;
  }
}

// Online-softmax update of one warp's 16 rows with one tile of up to 64 keys.
template <int HD, bool SPLIT>
DF_DEVICE void attend_tile(const uint32_t (&qh)[HD / 16][4], const uint32_t (&ql)[HD / 16][4],
                           const uint16_t* k_hi, const uint16_t* k_lo, const uint16_t* v_hi,
                           const uint16_t* v_lo, int KS, int nt, const int* kpos, bool blk, int p0,
                           int window, float& m0, float& m1, float& l0, float& l1,
                           float (&O)[HD / 8][4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  float S[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < nt) {
        const uint16_t* kr = k_hi + (8 * j + g) * KS + ks * 16 + 2 * t;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 8);
        mma_bf16_16816(S[j], qh[ks], b0, b1);
        mma_bf16_16816(S[j], ql[ks], b0, b1);
        if (SPLIT) {
          const uint16_t* kl = k_lo + (8 * j + g) * KS + ks * 16 + 2 * t;
          mma_bf16_16816(S[j], qh[ks], *reinterpret_cast<const uint32_t*>(kl),
                         *reinterpret_cast<const uint32_t*>(kl + 8));
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
        if (!blk) {
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
  const float c0 = m0 == -CUDART_INF_F ? 0.f : expf(m0 - n0);
  const float c1 = m1 == -CUDART_INF_F ? 0.f : expf(m1 - n1);
  m0 = n0;
  m1 = n1;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        S[j][e] = n0 == -CUDART_INF_F ? 0.f : expf(S[j][e] - n0);
        S[j][2 + e] = n1 == -CUDART_INF_F ? 0.f : expf(S[j][2 + e] - n1);
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
  const int lrow = lane & 7, lmat = lane >> 3;
#pragma unroll
  for (int jd = 0; jd < HD / 8; jd += 2) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (2 * kk < nt) {
        const int key = 16 * kk + (lmat & 1) * 8 + lrow;
        const int dim = 8 * jd + (lmat >> 1) * 8;
        uint32_t b[4];
        ldsm_x4_t(b, v_hi + key * KS + dim);
        mma_bf16_16816(O[jd], ph[kk], b[0], b[1]);
        mma_bf16_16816(O[jd], pl[kk], b[0], b[1]);
        mma_bf16_16816(O[jd + 1], ph[kk], b[2], b[3]);
        mma_bf16_16816(O[jd + 1], pl[kk], b[2], b[3]);
        if (SPLIT) {
          uint32_t bl[4];
          ldsm_x4_t(bl, v_lo + key * KS + dim);
          mma_bf16_16816(O[jd], ph[kk], bl[0], bl[1]);
          mma_bf16_16816(O[jd + 1], ph[kk], bl[2], bl[3]);
        }
      }
    }
  }
}

template <int HD, bool RING_F32>
__global__ void __launch_bounds__(256) attn_cluster_kernel(const __grid_constant__ AttnParams p) {
  using SM = AttnSmem<HD>;
  constexpr int KS = SM::KS;
  const int kDepth = p.depth;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const int kvh = blockIdx.y, seq = blockIdx.z;
  const int G = p.n_head / p.n_head_kv, R = kBlock * G;
  const int qd = p.n_head * HD, kvd = p.n_head_kv * HD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint16_t* bufs = reinterpret_cast<uint16_t*>(sm_raw);
  const int buf_elems = RING_F32 ? SM::BUF : 2 * SM::TILE;
  uint16_t* blk_k_hi = bufs + kDepth * buf_elems;
  uint16_t* blk_k_lo = blk_k_hi + kBlock * KS;
  uint16_t* blk_v_hi = blk_k_lo + kBlock * KS;
  uint16_t* blk_v_lo = blk_v_hi + kBlock * KS;
  int* kpos = reinterpret_cast<int*>(blk_v_lo + kBlock * KS);  // [kDepth][64]

  pdl_trigger();
  pdl_wait();
  const int p0 = max(p.n_past[seq], 0);
  const int per = (p.window + CL - 1) / CL;
  const int s_begin = min(p.window, rank * per), s_end = min(p.window, s_begin + per);
  const int n_sub = (s_end - s_begin + kSub - 1) / kSub;
  const size_t plane = (size_t)p.window * HD;
  const size_t kbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 0) * p.n_head_kv + kvh) * plane;
  const size_t vbase = kbase + (size_t)p.n_head_kv * plane;

  // async copy (bf16 ring) or load + split (fp32 ring) of ring sub-chunk j
  auto stage = [&](int j) {
    uint16_t* kh = bufs + (j % kDepth) * buf_elems;
    uint16_t* vh = kh + SM::TILE;
    uint16_t* kl = vh + SM::TILE;
    uint16_t* vl = kl + SM::TILE;
    const int s0 = s_begin + j * kSub, nk = min(kSub, s_end - s0);
    if (!RING_F32) {
      const uint16_t* r = reinterpret_cast<const uint16_t*>(p.ring);
      for (int idx = tid; idx < kSub * (HD / 8); idx += blockDim.x) {
        const int row = idx / (HD / 8), d = (idx - row * (HD / 8)) * 8;
        if (row < nk) {
          cp16(kh + row * KS + d, r + kbase + (size_t)(s0 + row) * HD + d);
          cp16(vh + row * KS + d, r + vbase + (size_t)(s0 + row) * HD + d);
        } else {
          *reinterpret_cast<uint4*>(kh + row * KS + d) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vh + row * KS + d) = make_uint4(0, 0, 0, 0);
        }
      }
    } else {
      const float* r = reinterpret_cast<const float*>(p.ring);
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
    int* kp = kpos + (j % kDepth) * kSub;
    for (int row = tid; row < kSub; row += blockDim.x)
      kp[row] = row < nk ? p.ring_pos[(size_t)seq * p.window + s0 + row] : -1;
    cp_commit();
  };

  for (int j = 0; j < kDepth - 1 && j < n_sub; ++j) stage(j);
  if (rank == 0) {  // the block's own 16 keys (fp32: split hi/lo)
    for (int idx = tid; idx < kBlock * (HD / 4); idx += blockDim.x) {
      const int row = idx / (HD / 4), d = (idx - row * (HD / 4)) * 4;
      const size_t o = (size_t)(seq * kBlock + row) * kvd + kvh * HD + d;
      const float4 kv = *reinterpret_cast<const float4*>(p.kblk + o);
      const float4 vv = *reinterpret_cast<const float4*>(p.vblk + o);
      uint2 h, l;
      split_bf16x2(kv.x, kv.y, h.x, l.x);
      split_bf16x2(kv.z, kv.w, h.y, l.y);
      *reinterpret_cast<uint2*>(blk_k_hi + row * KS + d) = h;
      *reinterpret_cast<uint2*>(blk_k_lo + row * KS + d) = l;
      split_bf16x2(vv.x, vv.y, h.x, l.x);
      split_bf16x2(vv.z, vv.w, h.y, l.y);
      *reinterpret_cast<uint2*>(blk_v_hi + row * KS + d) = h;
      *reinterpret_cast<uint2*>(blk_v_lo + row * KS + d) = l;
    }
  }

  // this warp's head: q fragments (fp32 -> scaled hi/lo) straight from global
  const bool active = warp < G;
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
  if (active) {
    const int head = kvh * G + warp;
    const float* qr0 = p.q + (size_t)(seq * kBlock + g) * qd + head * HD;
    const float* qr1 = qr0 + (size_t)8 * qd;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const int k0 = ks * 16 + 2 * t;
      const float2 a0 = *reinterpret_cast<const float2*>(qr0 + k0);
      const float2 a1 = *reinterpret_cast<const float2*>(qr1 + k0);
      const float2 a2 = *reinterpret_cast<const float2*>(qr0 + k0 + 8);
      const float2 a3 = *reinterpret_cast<const float2*>(qr1 + k0 + 8);
      split_bf16x2(a0.x * p.scale, a0.y * p.scale, qh[ks][0], ql[ks][0]);
      split_bf16x2(a1.x * p.scale, a1.y * p.scale, qh[ks][1], ql[ks][1]);
      split_bf16x2(a2.x * p.scale, a2.y * p.scale, qh[ks][2], ql[ks][2]);
      split_bf16x2(a3.x * p.scale, a3.y * p.scale, qh[ks][3], ql[ks][3]);
    }
  }
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float O[HD / 8][4];
#pragma unroll
  for (int jd = 0; jd < HD / 8; ++jd) O[jd][0] = O[jd][1] = O[jd][2] = O[jd][3] = 0.f;

  for (int j = 0; j < n_sub; ++j) {
    // keep kDepth - 1 sub-chunks in flight: issue j + kDepth - 1, wait for j
    if (j + kDepth - 1 < n_sub) stage(j + kDepth - 1);
    cp_wait_upto(min(kDepth - 1, n_sub - 1 - j));
    __syncthreads();
    if (active) {
      const uint16_t* kh = bufs + (j % kDepth) * buf_elems;
      attend_tile<HD, RING_F32>(qh, ql, kh, kh + 2 * SM::TILE, kh + SM::TILE, kh + 3 * SM::TILE, KS,
                                8, kpos + (j % kDepth) * kSub, false, p0, p.window, m0, m1, l0, l1, O,
                                lane);
    }
    __syncthreads();  // the buffer is refilled kDepth - 1 sub-chunks later
  }
  __syncthreads();
  if (rank == 0 && active)
    attend_tile<HD, true>(qh, ql, blk_k_hi, blk_k_lo, blk_v_hi, blk_v_lo, KS, 2, nullptr, true, p0,
                          p.window, m0, m1, l0, l1, O, lane);
  __syncthreads();

  // partials into this CTA's shared memory (over the K/V buffers), then merge
  float* part_o = reinterpret_cast<float*>(sm_raw);      // [R][HD]
  float2* part_ml = reinterpret_cast<float2*>(part_o + (size_t)R * HD);
  if (active) {
    float* o0 = part_o + (size_t)(warp * kBlock + g) * HD;
    float* o1 = o0 + (size_t)8 * HD;
#pragma unroll
    for (int jd = 0; jd < HD / 8; ++jd) {
      *reinterpret_cast<float2*>(o0 + 8 * jd + 2 * t) = make_float2(O[jd][0], O[jd][1]);
      *reinterpret_cast<float2*>(o1 + 8 * jd + 2 * t) = make_float2(O[jd][2], O[jd][3]);
    }
    if (t == 0) {
      part_ml[warp * kBlock + g] = make_float2(m0, l0);
      part_ml[warp * kBlock + g + 8] = make_float2(m1, l1);
    }
  }
  cluster.sync();
  const int rows_per = (R + CL - 1) / CL;
  const int r_lo = rank * rows_per, r_hi = min(R, r_lo + rows_per);
  const int nw = blockDim.x >> 5;
  for (int r = r_lo + warp; r < r_hi; r += nw) {
    // lane c < CL fetches rank c's (max, sum); the row's weights via shuffles
    float2 ml = make_float2(-CUDART_INF_F, 0.f);
    if (lane < CL) ml = cluster.map_shared_rank(part_ml, lane)[r];
    float M = ml.x;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wgt = (lane < CL && ml.x != -CUDART_INF_F) ? expf(ml.x - M) : 0.f;
    float L = wgt * ml.y;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    L = __shfl_sync(0xffffffffu, L, 0);  // lanes 0..7 hold the total
    float wc[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) wc[c] = __shfl_sync(0xffffffffu, wgt, c);
    // lane-parallel over dims, ranks summed in rank order
    for (int d = lane * 4; d < HD; d += 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) {
        if (c < CL) {
          const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(part_o, c) +
                                                             (size_t)r * HD + d);
          acc.x += wc[c] * v.x;
          acc.y += wc[c] * v.y;
          acc.z += wc[c] * v.z;
          acc.w += wc[c] * v.w;
        }
      }
      const float inv = 1.f / L;
      const float o4[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
      const int hl = r / kBlock, i = r - hl * kBlock;
      const size_t at = (size_t)(seq * kBlock + i) * qd + (kvh * G + hl) * HD + d;
      uint2 hi, lo;
      split_bf16x2(o4[0], o4[1], hi.x, lo.x);
      split_bf16x2(o4[2], o4[3], hi.y, lo.y);
      *reinterpret_cast<uint2*>(p.out_hi + at) = hi;
      *reinterpret_cast<uint2*>(p.out_lo + at) = lo;
    }
  }
  cluster.sync();  // peers may still be reading this CTA's partials
}

int attn_cluster_size(int window) {
  int cl = (window + 255) / 256;
  return cl < 1 ? 1 : (cl > kMaxCluster ? kMaxCluster : cl);
}

size_t attn_cluster_smem(int group, int hd, int ring_f32, int depth) {
  if (depth <= 0) depth = ring_f32 ? 2 : kMaxDepth;  // the largest the launcher picks
  size_t kv;
  switch (hd) {
    case 32: kv = AttnSmem<32>::bytes(ring_f32, depth); break;
    case 64: kv = AttnSmem<64>::bytes(ring_f32, depth); break;
    default: kv = AttnSmem<128>::bytes(ring_f32, depth); break;
  }
  const size_t part = (size_t)kBlock * group * hd * 4 + (size_t)kBlock * group * 8;
  return kv > part ? kv : part;
}

template <int HD, bool F32>
static cudaError_t configure_cl(size_t smem) {
  static size_t configured = 0;   // only ever raised, so every live handle still fits
  if (smem <= configured) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<HD, F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) configured = smem;
  return e;
}

cudaError_t configure_attention_cluster(int group, int hd, int ring_f32) {
  const size_t smem = attn_cluster_smem(group, hd, ring_f32, 0);
  switch (hd) {
    case 32: return ring_f32 ? configure_cl<32, true>(smem) : configure_cl<32, false>(smem);
    case 64: return ring_f32 ? configure_cl<64, true>(smem) : configure_cl<64, false>(smem);
    case 128: return ring_f32 ? configure_cl<128, true>(smem) : configure_cl<128, false>(smem);
  }
  return cudaErrorInvalidValue;
}

template <int HD, bool F32>
static cudaError_t launch_cl(const AttnParams& p_in, int n_seq, cudaStream_t st) {
  const int G = p_in.n_head / p_in.n_head_kv, CL = attn_cluster_size(p_in.window);
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (n_sm <= 0) n_sm = 1;
  }
  AttnParams p = p_in;
  p.depth = depth_for(F32, (long long)CL * p.n_head_kv * n_seq, n_sm);
  const size_t smem = attn_cluster_smem(G, HD, F32, p.depth);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, p.n_head_kv, n_seq);
  cfg.blockDim = dim3(32 * G);
  cfg.dynamicSmemBytes = smem;
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

}  // namespace dflash
