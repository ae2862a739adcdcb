// Non-GEMM kernels of the drafter step: block embedding + rope tables,
// sliding-window GQA attention split over ring chunks, its combine, the
// RMSNorm apply of encode, and the first-mismatch acceptance scan.
#include "common.cuh"
#include "internal.h"

#include <math_constants.h>

namespace dflash {

// ------------------------------------------------------------------ embedding

// Block rows: token id_last for row 0, mask_token for rows 1..15 (dflash-ops model
// card, Method; dflash_head.rs field mask_token_id).  Writes h (fp32) and the
// row's sum of squares for the first layer's RMSNorm.  Extra blocks fill the
// rope table of the block positions n_past + i from the host fp64
// inverse-frequency table (angle and sin/cos in fp64, then rounded to fp32).
__global__ void __launch_bounds__(256) embed_kernel(const void* tok_embd, int dense_bf16, int d,
                                                    int V, int mask_token, const int32_t* id_last,
                                                    const int32_t* n_past, int n_seq,
                                                    const double* inv_freq, int half, float* h,
                                                    float* ss, float2* rope_cs, const void* norm0,
                                                    uint16_t* x_hi, uint16_t* x_lo,
                                                    unsigned* status) {
  const int M = n_seq * kBlock;
  if ((int)blockIdx.x < M) {
    const int m = blockIdx.x, seq = m / kBlock, i = m % kBlock;
    int tok = i == 0 ? id_last[seq] : mask_token;
    if (tok < 0 || tok >= V) {
      if (threadIdx.x == 0) atomicOr(status, 0x1u);
      tok = tok < 0 ? 0 : V - 1;
    }
    // 8 elements per thread and round (one 16-byte bf16 load or two float4
    // loads), all loads of a round issued before any store
    float s = 0.f;
    constexpr int kRound = 4;
    for (int k0 = threadIdx.x * 8; k0 < d; k0 += kRound * (int)blockDim.x * 8) {
      float v[kRound][8];
#pragma unroll
      for (int r = 0; r < kRound; ++r) {
        const int k = k0 + r * blockDim.x * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) v[r][e] = 0.f;
        if (k >= d) continue;
        if (dense_bf16) {
          const uint4 b = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(tok_embd) +
                                                         (size_t)tok * d + k);
          const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[r][2 * e] = __uint_as_float(w[e] << 16);
            v[r][2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
        } else {
          const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(tok_embd) +
                                                              (size_t)tok * d + k);
          const float4 a = src[0], b = src[1];
          v[r][0] = a.x; v[r][1] = a.y; v[r][2] = a.z; v[r][3] = a.w;
          v[r][4] = b.x; v[r][5] = b.y; v[r][6] = b.z; v[r][7] = b.w;
        }
      }
#pragma unroll
      for (int r = 0; r < kRound; ++r) {
        const int k = k0 + r * blockDim.x * 8;
        if (k >= d) continue;
        float4* dst = reinterpret_cast<float4*>(h + (size_t)m * d + k);
        dst[0] = make_float4(v[r][0], v[r][1], v[r][2], v[r][3]);
        dst[1] = make_float4(v[r][4], v[r][5], v[r][6], v[r][7]);
        // first layer's projection input: h * attn_norm, split into bf16 hi + lo
        uint32_t hh[4], ll[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float z0 = v[r][2 * e] * load_dense(norm0, dense_bf16, k + 2 * e);
          const float z1 = v[r][2 * e + 1] * load_dense(norm0, dense_bf16, k + 2 * e + 1);
          split_bf16x2(z0, z1, hh[e], ll[e]);
        }
        *reinterpret_cast<uint4*>(x_hi + (size_t)m * d + k) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
        *reinterpret_cast<uint4*>(x_lo + (size_t)m * d + k) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += v[r][e] * v[r][e];
      }
    }
    __shared__ float red[8];
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
      ss[m] = t;
    }
    return;
  }
  const int e = (blockIdx.x - M) * blockDim.x + threadIdx.x;
  if (e >= M * half) return;
  const int m = e / half, j = e - m * half, seq = m / kBlock;
  int p0 = n_past[seq];
  if (p0 < 0) {
    atomicOr(status, 0x2u);
    p0 = 0;
  }
  double sn, cs;
  sincos((double)(p0 + (m % kBlock)) * inv_freq[j], &sn, &cs);
  rope_cs[e] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_embed(const void* tok_embd, int dense_bf16, int n_embd, int n_vocab,
                         int mask_token, const int32_t* id_last, const int32_t* n_past, int n_seq,
                         const double* inv_freq, int hd, float* h, float* ss, float2* rope_cs,
                         const void* norm0, uint16_t* x_hi, uint16_t* x_lo, unsigned* status,
                         cudaStream_t st) {
  const int M = n_seq * kBlock, half = hd / 2;
  const int tb = (M * half + 255) / 256;
  embed_kernel<<<M + tb, 256, 0, st>>>(tok_embd, dense_bf16, n_embd, n_vocab, mask_token, id_last,
                                       n_past, n_seq, inv_freq, half, h, ss, rope_cs, norm0, x_hi,
                                       x_lo, status);
  return cudaGetLastError();
}

// Rope table of injected positions + ring_pos of their slots.
__global__ void rope_table_kernel(const int32_t* pos, int T, const double* inv_freq, int half,
                                  float2* rope_cs, int32_t* ring_pos, int window,
                                  unsigned* status) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= T * half) return;
  const int t = e / half, j = e - t * half;
  int p = pos[t];
  if (p < 0) {
    if (j == 0) atomicOr(status, 0x2u);
    p = 0;
  } else if (j == 0) {
    ring_pos[p % window] = p;
  }
  double sn, cs;
  sincos((double)p * inv_freq[j], &sn, &cs);
  rope_cs[e] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(const int32_t* pos, int T, const double* inv_freq, int hd,
                              float2* rope_cs, int32_t* ring_pos, int window, unsigned* status,
                              cudaStream_t st) {
  const int half = hd / 2;
  if (T <= 0) return cudaSuccess;
  rope_table_kernel<<<(T * half + 255) / 256, 256, 0, st>>>(pos, T, inv_freq, half, rope_cs,
                                                            ring_pos, window, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ RMSNorm apply

__global__ void __launch_bounds__(256) rms_apply_kernel(const float* raw, const float* ss, int n_ss,
                                                        int ss_ld, int n, const void* normw,
                                                        int norm_bf16, float eps, float* out) {
  const int t = blockIdx.x;
  __shared__ float inv;
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int q = 0; q < n_ss; ++q) s += ss[(size_t)q * ss_ld + t];
    inv = 1.f / sqrtf(s / (float)n + eps);
  }
  __syncthreads();
  for (int k = threadIdx.x; k < n; k += blockDim.x)
    out[(size_t)t * n + k] = raw[(size_t)t * n + k] * inv * load_dense(normw, norm_bf16, k);
}

cudaError_t launch_rms_apply(const float* raw, const float* ss, int n_ss, int ss_ld, int T, int n,
                             const void* normw, int norm_bf16, float eps, float* out,
                             cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  rms_apply_kernel<<<T, 256, 0, st>>>(raw, ss, n_ss, ss_ld, n, normw, norm_bf16, eps, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ attention

// One CTA = one (sequence, kv head, key chunk); one warp per query head of the
// kv group (16 block rows each), all warps sharing the chunk's K/V tile in
// shared memory.  Chunk c < n_chunks covers ring slots [c*64, c*64 + 64);
// chunk n_chunks is the block's own 16 keys, visible to every row
// (non-causal).  A ring slot holding position kp is a key of row i iff
// 0 <= kp < n_past and (n_past + i) - kp < window (dflash-ops model card,
// Method).  Both products run on the tensor cores with fp32 accumulation:
// q (fp32, pre-scaled by 1/sqrt(hd)) and the probabilities p (fp32) are split
// into bf16 hi + lo; bf16 ring K/V are exact, fp32 K/V (an fp32 ring, or the
// block's own keys) are split too, so S = q k^T and O = p V keep fp32
// accuracy (~2^-17 per product).  Each CTA writes the chunk's row max, row sum
// of exp and unnormalised O for the merge kernel.
constexpr int kAttnChunk = 64;
constexpr int kKPad = 8;   // bf16 elements of row padding (16 B): conflict-free fragment loads

DF_DEVICE void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
DF_DEVICE void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// four 8x8 bf16 matrices, transposed on the way out (B fragments of p V)
DF_DEVICE void ldmatrix_x4_trans(uint32_t (&r)[4], const void* smem) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

template <int HD>
__global__ void attn_chunk_kernel(const __grid_constant__ AttnParams p) {
  constexpr int KS = HD + kKPad;     // row stride of K / V tiles (bf16 elements)
  constexpr int NK16 = HD / 16;      // k16 steps over the head dimension
  const int c = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int G = p.n_head / p.n_head_kv;
  const int qd = p.n_head * HD, kvd = p.n_head_kv * HD;
  const bool blk = c == p.n_chunks;
  const int s0 = c * kAttnChunk;
  const int nk = blk ? kBlock : min(kAttnChunk, p.window - s0);
  const bool split_kv = blk || !p.ring_bf16;     // K/V arrive as fp32 -> hi + lo
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint16_t* k_hi = reinterpret_cast<uint16_t*>(sm_raw);   // [64][KS]
  uint16_t* k_lo = k_hi + kAttnChunk * KS;
  uint16_t* v_hi = k_lo + kAttnChunk * KS;                // [64][KS] (row-major, keys x dims)
  uint16_t* v_lo = v_hi + kAttnChunk * KS;
  int* kpos = reinterpret_cast<int*>(v_lo + kAttnChunk * KS);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;

  pdl_trigger();
  pdl_wait();
  const int p0 = max(p.n_past[seq], 0);

  // K/V tile: bf16 ring rows by 16-byte async copies; fp32 rows split hi/lo
  const size_t plane = (size_t)p.window * HD;
  const size_t kbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 0) * p.n_head_kv + kvh) * plane;
  const size_t vbase = kbase + (size_t)p.n_head_kv * plane;
  if (!split_kv) {
    const uint16_t* r = reinterpret_cast<const uint16_t*>(p.ring);
    for (int idx = tid; idx < kAttnChunk * (HD / 8); idx += blockDim.x) {
      const int j = idx / (HD / 8), d = (idx - j * (HD / 8)) * 8;
      if (j < nk) {
        cp_async16(k_hi + j * KS + d, r + kbase + (size_t)(s0 + j) * HD + d);
        cp_async16(v_hi + j * KS + d, r + vbase + (size_t)(s0 + j) * HD + d);
      } else {
        *reinterpret_cast<uint4*>(k_hi + j * KS + d) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(v_hi + j * KS + d) = make_uint4(0, 0, 0, 0);
      }
    }
  } else {
    const int rows = blk ? kBlock : kAttnChunk;
    for (int idx = tid; idx < rows * (HD / 4); idx += blockDim.x) {
      const int j = idx / (HD / 4), d = (idx - j * (HD / 4)) * 4;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (j < nk) {
        if (blk) {
          const size_t o = (size_t)(seq * kBlock + j) * kvd + kvh * HD + d;
          kv = *reinterpret_cast<const float4*>(p.kblk + o);
          vv = *reinterpret_cast<const float4*>(p.vblk + o);
        } else {
          const float* r = reinterpret_cast<const float*>(p.ring);
          kv = *reinterpret_cast<const float4*>(r + kbase + (size_t)(s0 + j) * HD + d);
          vv = *reinterpret_cast<const float4*>(r + vbase + (size_t)(s0 + j) * HD + d);
        }
      }
      uint2 h, l;
      split_bf16x2(kv.x, kv.y, h.x, l.x);
      split_bf16x2(kv.z, kv.w, h.y, l.y);
      *reinterpret_cast<uint2*>(k_hi + j * KS + d) = h;
      *reinterpret_cast<uint2*>(k_lo + j * KS + d) = l;
      split_bf16x2(vv.x, vv.y, h.x, l.x);
      split_bf16x2(vv.z, vv.w, h.y, l.y);
      *reinterpret_cast<uint2*>(v_hi + j * KS + d) = h;
      *reinterpret_cast<uint2*>(v_lo + j * KS + d) = l;
    }
  }
  for (int j = tid; j < kAttnChunk; j += blockDim.x)
    kpos[j] = (blk || j >= nk) ? -1 : p.ring_pos[(size_t)seq * p.window + s0 + j];

  // q fragments of this warp's head straight from global (fp32 -> hi/lo), while
  // the K/V copies are in flight
  const int head = kvh * G + warp;
  const float* qrow0 = p.q + (size_t)(seq * kBlock + g) * qd + head * HD;
  const float* qrow1 = qrow0 + (size_t)8 * qd;
  uint32_t qh[NK16][4], ql[NK16][4];
#pragma unroll
  for (int ks = 0; ks < NK16; ++ks) {
    const int k0 = ks * 16 + 2 * t;
    const float2 a0 = *reinterpret_cast<const float2*>(qrow0 + k0);
    const float2 a1 = *reinterpret_cast<const float2*>(qrow1 + k0);
    const float2 a2 = *reinterpret_cast<const float2*>(qrow0 + k0 + 8);
    const float2 a3 = *reinterpret_cast<const float2*>(qrow1 + k0 + 8);
    split_bf16x2(a0.x * p.scale, a0.y * p.scale, qh[ks][0], ql[ks][0]);
    split_bf16x2(a1.x * p.scale, a1.y * p.scale, qh[ks][1], ql[ks][1]);
    split_bf16x2(a2.x * p.scale, a2.y * p.scale, qh[ks][2], ql[ks][2]);
    split_bf16x2(a3.x * p.scale, a3.y * p.scale, qh[ks][3], ql[ks][3]);
  }
  cp_async_wait_all();
  __syncthreads();

  // S = q k^T: 16 rows x up to 64 keys (8 n8 tiles)
  const int nt = blk ? 2 : 8;
  float S[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < NK16; ++ks) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < nt) {
        const uint16_t* kr = k_hi + (8 * j + g) * KS + ks * 16 + 2 * t;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 8);
        mma_bf16_16816(S[j], qh[ks], b0, b1);
        mma_bf16_16816(S[j], ql[ks], b0, b1);
        if (split_kv) {
          const uint16_t* kl = k_lo + (8 * j + g) * KS + ks * 16 + 2 * t;
          mma_bf16_16816(S[j], qh[ks], *reinterpret_cast<const uint32_t*>(kl),
                         *reinterpret_cast<const uint32_t*>(kl + 8));
        }
      }
    }
  }
  // mask, row max, exp, row sum (rows g and g + 8; a row lives in one lane quad)
  const int qpos0 = p0 + g, qpos1 = p0 + g + 8;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = 8 * j + 2 * t + e;
        bool ok0 = true, ok1 = true;
        if (!blk) {
          const int kp = kpos[key];
          const bool past = kp >= 0 && kp < p0;
          ok0 = past && qpos0 - kp < p.window;
          ok1 = past && qpos1 - kp < p.window;
        }
        if (!ok0) S[j][e] = -CUDART_INF_F;
        if (!ok1) S[j][2 + e] = -CUDART_INF_F;
        m0 = fmaxf(m0, S[j][e]);
        m1 = fmaxf(m1, S[j][2 + e]);
      }
    }
  }
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        S[j][e] = m0 == -CUDART_INF_F ? 0.f : expf(S[j][e] - m0);
        S[j][2 + e] = m1 == -CUDART_INF_F ? 0.f : expf(S[j][2 + e] - m1);
        l0 += S[j][e];
        l1 += S[j][2 + e];
      }
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // O = p V: p from the S accumulators (two key n8 tiles = one k16 step); the
  // V fragments come from the row-major tile through ldmatrix.trans
  uint32_t ph[4][4], pl[4][4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    split_bf16x2(S[2 * kk][0], S[2 * kk][1], ph[kk][0], pl[kk][0]);
    split_bf16x2(S[2 * kk][2], S[2 * kk][3], ph[kk][1], pl[kk][1]);
    split_bf16x2(S[2 * kk + 1][0], S[2 * kk + 1][1], ph[kk][2], pl[kk][2]);
    split_bf16x2(S[2 * kk + 1][2], S[2 * kk + 1][3], ph[kk][3], pl[kk][3]);
  }
  const size_t slot = ((size_t)seq * p.n_head_kv + kvh) * (p.n_chunks + 1) + c;
  const int R = kBlock * G;
  float* oacc = p.part_acc + (slot * R + warp * kBlock) * HD;
  // lane -> row of the 8x8 matrix it addresses for ldmatrix: matrices 0/1 are
  // keys [0,8) / [8,16) of dims [8jd, 8jd+8), matrices 2/3 the next 8 dims
  const int lrow = lane & 7, lmat = lane >> 3;
#pragma unroll
  for (int jd = 0; jd < HD / 8; jd += 2) {
    float O0[4] = {0.f, 0.f, 0.f, 0.f}, O1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (2 * kk < nt) {
        const int key = 16 * kk + (lmat & 1) * 8 + lrow;
        const int dim = 8 * jd + (lmat >> 1) * 8;
        uint32_t b[4];
        ldmatrix_x4_trans(b, v_hi + key * KS + dim);
        mma_bf16_16816(O0, ph[kk], b[0], b[1]);
        mma_bf16_16816(O0, pl[kk], b[0], b[1]);
        mma_bf16_16816(O1, ph[kk], b[2], b[3]);
        mma_bf16_16816(O1, pl[kk], b[2], b[3]);
        if (split_kv) {
          uint32_t bl[4];
          ldmatrix_x4_trans(bl, v_lo + key * KS + dim);
          mma_bf16_16816(O0, ph[kk], bl[0], bl[1]);
          mma_bf16_16816(O1, ph[kk], bl[2], bl[3]);
        }
      }
    }
    *reinterpret_cast<float2*>(oacc + (size_t)g * HD + 8 * jd + 2 * t) = make_float2(O0[0], O0[1]);
    *reinterpret_cast<float2*>(oacc + (size_t)(g + 8) * HD + 8 * jd + 2 * t) = make_float2(O0[2], O0[3]);
    *reinterpret_cast<float2*>(oacc + (size_t)g * HD + 8 * jd + 8 + 2 * t) = make_float2(O1[0], O1[1]);
    *reinterpret_cast<float2*>(oacc + (size_t)(g + 8) * HD + 8 * jd + 8 + 2 * t) = make_float2(O1[2], O1[3]);
  }
  if (t == 0) {
    float* ml = p.part_ml + (slot * R + warp * kBlock) * 2;
    ml[g * 2 + 0] = m0;
    ml[g * 2 + 1] = l0;
    ml[(g + 8) * 2 + 0] = m1;
    ml[(g + 8) * 2 + 1] = l1;
  }
}

size_t attn_smem_bytes(int group, int hd, int ring_f32) {
  (void)group;
  (void)ring_f32;
  return sizeof(uint16_t) * 4 * (size_t)kAttnChunk * (hd + kKPad) + sizeof(int) * kAttnChunk;
}

cudaError_t configure_attention(size_t smem) {
  static size_t configured = 0;   // only ever raised, so every live handle still fits
  if (smem <= configured) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel<32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_chunk_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_chunk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (e == cudaSuccess) configured = smem;
  return e;
}

static cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t launch_attention(const AttnParams& p, int n_seq, cudaStream_t st) {
  const int G = p.n_head / p.n_head_kv;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.n_chunks + 1, p.n_head_kv, n_seq), dim3(32 * G),
                                      attn_smem_bytes(G, p.hd, !p.ring_bf16), st, attr);
  switch (p.hd) {
    case 32: return cudaLaunchKernelEx(&cfg, attn_chunk_kernel<32>, p);
    case 64: return cudaLaunchKernelEx(&cfg, attn_chunk_kernel<64>, p);
    case 128: return cudaLaunchKernelEx(&cfg, attn_chunk_kernel<128>, p);
  }
  return cudaErrorInvalidValue;
}

// Merge the chunk partials of one (sequence, query head, 4 block rows) in chunk
// order: out = sum_c exp(m_c - M) O_c / sum_c exp(m_c - M) l_c.  One thread per
// (row, dim); the chunk loops issue independent loads.
constexpr int kMergeRows = 4;

__global__ void __launch_bounds__(512) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  pdl_trigger();
  pdl_wait();
  const int per_head = kBlock / kMergeRows;
  const int rb = blockIdx.x % per_head, h = (blockIdx.x / per_head) % p.n_head;
  const int seq = blockIdx.x / (per_head * p.n_head);
  const int G = p.n_head / p.n_head_kv, kvh = h / G, hl = h - kvh * G;
  const int R = kBlock * G, hd = p.hd, nc = p.n_chunks + 1;
  const int i = rb * kMergeRows + threadIdx.x / hd, d = threadIdx.x % hd;
  if (threadIdx.x >= kMergeRows * hd) return;
  const int r = hl * kBlock + i;
  const size_t slot0 = ((size_t)seq * p.n_head_kv + kvh) * nc;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  float M = -CUDART_INF_F;
#pragma unroll 8
  for (int c = 0; c < nc; ++c) M = fmaxf(M, ml[(slot0 + c) * R + r].x);
  float L = 0.f, A = 0.f;
#pragma unroll 8
  for (int c = 0; c < nc; ++c) {
    const float2 e = ml[(slot0 + c) * R + r];
    const float o = p.part_acc[((slot0 + c) * R + r) * hd + d];
    const float w = e.x == -CUDART_INF_F ? 0.f : expf(e.x - M);
    L += e.y * w;
    A += o * w;
  }
  const float o = A / L;
  const size_t at = (size_t)(seq * kBlock + i) * (p.n_head * hd) + h * hd + d;
  const uint16_t oh = f32_to_bf16_bits(o);
  p.out_hi[at] = oh;
  p.out_lo[at] = f32_to_bf16_bits(o - bf16_bits_to_f32(oh));
}

cudaError_t launch_attn_combine(const AttnParams& p, int n_seq, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(n_seq * p.n_head * (kBlock / kMergeRows)),
                                      dim3(kMergeRows * p.hd), 0, st, attr);
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, p);
}

// ------------------------------------------------------------------ acceptance

// One warp per sequence: lanes 0..14 compare draft j with the target's token j,
// a ballot marks the mismatches, and the first set bit is the number of leading
// matches (15 when none): dflash-ops model card, Usage (device-side accept) and
// dflash_engine.py, DFlashSpeculativeVerifier.verify_block.
__global__ void accept_kernel(const int32_t* drafts, const int32_t* targets, int32_t* n_ok,
                              int n_seq) {
  const int seq = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (seq >= n_seq) return;
  bool miss = false;
  if (lane < kBlock - 1) miss = drafts[seq * (kBlock - 1) + lane] != targets[seq * (kBlock - 1) + lane];
  const unsigned mask = __ballot_sync(0xffffffffu, miss);
  if (lane == 0) n_ok[seq] = mask ? __ffs(mask) - 1 : kBlock - 1;
}

cudaError_t launch_accept(const int32_t* drafts, const int32_t* targets, int32_t* n_ok, int n_seq,
                          cudaStream_t st) {
  accept_kernel<<<(n_seq + 7) / 8, 256, 0, st>>>(drafts, targets, n_ok, n_seq);
  return cudaGetLastError();
}

__global__ void fill_i32_kernel(int32_t* p, int n, int32_t v) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

cudaError_t launch_fill_i32(int32_t* p, int n, int32_t v, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  fill_i32_kernel<<<(n + 255) / 256, 256, 0, st>>>(p, n, v);
  return cudaGetLastError();
}

}  // namespace dflash
