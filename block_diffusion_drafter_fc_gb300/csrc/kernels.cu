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
                                                    float* ss, float2* rope_cs, unsigned* status) {
  const int M = n_seq * kBlock;
  if ((int)blockIdx.x < M) {
    const int m = blockIdx.x, seq = m / kBlock, i = m % kBlock;
    int tok = i == 0 ? id_last[seq] : mask_token;
    if (tok < 0 || tok >= V) {
      if (threadIdx.x == 0) atomicOr(status, 0x1u);
      tok = tok < 0 ? 0 : V - 1;
    }
    float s = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
      const float v = load_dense(tok_embd, dense_bf16, (size_t)tok * d + k);
      h[(size_t)m * d + k] = v;
      s += v * v;
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
                         unsigned* status, cudaStream_t st) {
  const int M = n_seq * kBlock, half = hd / 2;
  const int tb = (M * half + 255) / 256;
  embed_kernel<<<M + tb, 256, 0, st>>>(tok_embd, dense_bf16, n_embd, n_vocab, mask_token, id_last,
                                       n_past, n_seq, inv_freq, half, h, ss, rope_cs, status);
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
// into bf16 hi + lo, bf16 ring K/V are exact (an fp32 ring is split too), so
// S = q k^T and O = p V keep fp32 accuracy (~2^-17 per product).  Each CTA
// writes the chunk's row max, row sum of exp and unnormalised O.
constexpr int kAttnChunk = 64;
constexpr int kQPad = 8, kVPad = 8;

template <bool RING_F32>
__global__ void attn_chunk_kernel(const __grid_constant__ AttnParams p) {
  const int c = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int G = p.n_head / p.n_head_kv, R = kBlock * G, hd = p.hd;
  const int qd = p.n_head * hd, kvd = p.n_head_kv * hd;
  const bool blk = c == p.n_chunks;
  const int s0 = c * kAttnChunk;
  const int CH = blk ? kBlock : kAttnChunk;               // keys in this tile (padded)
  const int nk = blk ? kBlock : min(kAttnChunk, p.window - s0);
  const int QS = hd + kQPad, VS = kAttnChunk + kVPad;
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint16_t* q_hi = reinterpret_cast<uint16_t*>(sm_raw);   // [R][QS]
  uint16_t* q_lo = q_hi + R * QS;
  uint16_t* k_hi = q_lo + R * QS;                         // [64][QS]
  uint16_t* k_lo = k_hi + kAttnChunk * QS;
  uint16_t* v_hi = k_lo + (RING_F32 ? kAttnChunk * QS : 0);  // transposed [hd][VS]
  uint16_t* v_lo = v_hi + hd * VS;
  int* kpos = reinterpret_cast<int*>(v_lo + (RING_F32 ? hd * VS : 0));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;

  pdl_trigger();
  pdl_wait();
  const int p0 = max(p.n_past[seq], 0);

  // q rows of the group (row r = head_local * 16 + i), scaled, split hi/lo
  for (int idx = tid; idx < R * hd / 4; idx += blockDim.x) {
    const int r = idx / (hd / 4), d = (idx - r * (hd / 4)) * 4;
    const int hl = r / kBlock, i = r - hl * kBlock;
    float4 v = *reinterpret_cast<const float4*>(p.q + (size_t)(seq * kBlock + i) * qd + (kvh * G + hl) * hd + d);
    v.x *= p.scale; v.y *= p.scale; v.z *= p.scale; v.w *= p.scale;
    uint2 h, l;
    split_bf16x2(v.x, v.y, h.x, l.x);
    split_bf16x2(v.z, v.w, h.y, l.y);
    *reinterpret_cast<uint2*>(q_hi + r * QS + d) = h;
    *reinterpret_cast<uint2*>(q_lo + r * QS + d) = l;
  }
  // keys / values of the chunk (rows past nk are zero and masked)
  const size_t plane = (size_t)p.window * hd;
  const size_t kbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 0) * p.n_head_kv + kvh) * plane;
  const size_t vbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 1) * p.n_head_kv + kvh) * plane;
  for (int idx = tid; idx < CH * hd / 4; idx += blockDim.x) {
    const int j = idx / (hd / 4), d = (idx - j * (hd / 4)) * 4;
    float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
    if (j < nk) {
      if (blk) {
        const size_t o = (size_t)(seq * kBlock + j) * kvd + kvh * hd + d;
        kv = *reinterpret_cast<const float4*>(p.kblk + o);
        vv = *reinterpret_cast<const float4*>(p.vblk + o);
      } else if (RING_F32) {
        const float* r = reinterpret_cast<const float*>(p.ring);
        kv = *reinterpret_cast<const float4*>(r + kbase + (size_t)(s0 + j) * hd + d);
        vv = *reinterpret_cast<const float4*>(r + vbase + (size_t)(s0 + j) * hd + d);
      } else {
        const uint16_t* r = reinterpret_cast<const uint16_t*>(p.ring);
        const uint2 kb = *reinterpret_cast<const uint2*>(r + kbase + (size_t)(s0 + j) * hd + d);
        const uint2 vb = *reinterpret_cast<const uint2*>(r + vbase + (size_t)(s0 + j) * hd + d);
        kv = make_float4(__uint_as_float(kb.x << 16), __uint_as_float(kb.x & 0xffff0000u),
                         __uint_as_float(kb.y << 16), __uint_as_float(kb.y & 0xffff0000u));
        vv = make_float4(__uint_as_float(vb.x << 16), __uint_as_float(vb.x & 0xffff0000u),
                         __uint_as_float(vb.y << 16), __uint_as_float(vb.y & 0xffff0000u));
      }
    }
    uint2 kh, kl;
    split_bf16x2(kv.x, kv.y, kh.x, kl.x);
    split_bf16x2(kv.z, kv.w, kh.y, kl.y);
    *reinterpret_cast<uint2*>(k_hi + j * QS + d) = kh;
    if (RING_F32) *reinterpret_cast<uint2*>(k_lo + j * QS + d) = kl;
    const float va[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint16_t vh = f32_to_bf16_bits(va[e]);
      v_hi[(d + e) * VS + j] = vh;
      if (RING_F32) v_lo[(d + e) * VS + j] = f32_to_bf16_bits(va[e] - bf16_bits_to_f32(vh));
    }
  }
  for (int j = tid; j < CH; j += blockDim.x)
    kpos[j] = (blk || j >= nk) ? -1 : p.ring_pos[(size_t)seq * p.window + s0 + j];
  __syncthreads();
  if (warp >= G) return;

  // S = q k^T for this warp's 16 rows (head `warp`) and up to 64 keys
  const uint16_t* qh = q_hi + warp * kBlock * QS;
  const uint16_t* ql = q_lo + warp * kBlock * QS;
  float S[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
  const int nt = CH / 8;
  for (int k0 = 0; k0 < hd; k0 += 16) {
    const uint32_t ah[4] = {*reinterpret_cast<const uint32_t*>(qh + g * QS + k0 + 2 * t),
                            *reinterpret_cast<const uint32_t*>(qh + (g + 8) * QS + k0 + 2 * t),
                            *reinterpret_cast<const uint32_t*>(qh + g * QS + k0 + 2 * t + 8),
                            *reinterpret_cast<const uint32_t*>(qh + (g + 8) * QS + k0 + 2 * t + 8)};
    const uint32_t al[4] = {*reinterpret_cast<const uint32_t*>(ql + g * QS + k0 + 2 * t),
                            *reinterpret_cast<const uint32_t*>(ql + (g + 8) * QS + k0 + 2 * t),
                            *reinterpret_cast<const uint32_t*>(ql + g * QS + k0 + 2 * t + 8),
                            *reinterpret_cast<const uint32_t*>(ql + (g + 8) * QS + k0 + 2 * t + 8)};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= nt) break;
      const uint16_t* kr = k_hi + (8 * j + g) * QS + k0 + 2 * t;
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 8);
      mma_bf16_16816(S[j], ah, b0, b1);
      mma_bf16_16816(S[j], al, b0, b1);
      if (RING_F32) {
        const uint16_t* kl2 = k_lo + (8 * j + g) * QS + k0 + 2 * t;
        mma_bf16_16816(S[j], ah, *reinterpret_cast<const uint32_t*>(kl2),
                       *reinterpret_cast<const uint32_t*>(kl2 + 8));
      }
    }
  }
  // mask, row max, exp, row sum (rows g and g + 8; a row lives in one lane quad)
  const int qpos0 = p0 + g, qpos1 = p0 + g + 8;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= nt) break;
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
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= nt) break;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      S[j][e] = m0 == -CUDART_INF_F ? 0.f : expf(S[j][e] - m0);
      S[j][2 + e] = m1 == -CUDART_INF_F ? 0.f : expf(S[j][2 + e] - m1);
      l0 += S[j][e];
      l1 += S[j][2 + e];
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // O = p V: p from the S accumulators (two key n8 tiles = one k16 step)
  const size_t slot = ((size_t)seq * p.n_head_kv + kvh) * (p.n_chunks + 1) + c;
  float* oacc = p.part_acc + (slot * R + warp * kBlock) * hd;
  for (int jd = 0; jd < hd / 8; ++jd) {
    float O[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (2 * kk >= nt) break;
      uint32_t ph[4], pl[4];
      split_bf16x2(S[2 * kk][0], S[2 * kk][1], ph[0], pl[0]);
      split_bf16x2(S[2 * kk][2], S[2 * kk][3], ph[1], pl[1]);
      split_bf16x2(S[2 * kk + 1][0], S[2 * kk + 1][1], ph[2], pl[2]);
      split_bf16x2(S[2 * kk + 1][2], S[2 * kk + 1][3], ph[3], pl[3]);
      const uint16_t* vr = v_hi + (8 * jd + g) * VS + 16 * kk + 2 * t;
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(vr);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(vr + 8);
      mma_bf16_16816(O, ph, b0, b1);
      mma_bf16_16816(O, pl, b0, b1);
      if (RING_F32) {
        const uint16_t* vl = v_lo + (8 * jd + g) * VS + 16 * kk + 2 * t;
        mma_bf16_16816(O, ph, *reinterpret_cast<const uint32_t*>(vl),
                       *reinterpret_cast<const uint32_t*>(vl + 8));
      }
    }
    *reinterpret_cast<float2*>(oacc + (size_t)g * hd + 8 * jd + 2 * t) = make_float2(O[0], O[1]);
    *reinterpret_cast<float2*>(oacc + (size_t)(g + 8) * hd + 8 * jd + 2 * t) = make_float2(O[2], O[3]);
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
  const int R = kBlock * group, QS = hd + kQPad, VS = kAttnChunk + kVPad;
  size_t b = sizeof(uint16_t) * (2 * (size_t)R * QS + (size_t)kAttnChunk * QS + (size_t)hd * VS);
  if (ring_f32) b += sizeof(uint16_t) * ((size_t)kAttnChunk * QS + (size_t)hd * VS);
  return b + sizeof(int) * kAttnChunk;
}

cudaError_t configure_attention(size_t smem) {
  static size_t configured = 0;   // only ever raised, so every live handle still fits
  if (smem <= configured) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_chunk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t launch_attention(const AttnParams& p, int n_seq, cudaStream_t st) {
  const int G = p.n_head / p.n_head_kv;
  const int f32 = !p.ring_bf16;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.n_chunks + 1, p.n_head_kv, n_seq),
                                      dim3(32 * G),
                                      attn_smem_bytes(G, p.hd, f32), st, attr);
  return f32 ? cudaLaunchKernelEx(&cfg, attn_chunk_kernel<true>, p)
             : cudaLaunchKernelEx(&cfg, attn_chunk_kernel<false>, p);
}

// Merge the chunk partials of one (sequence, query head) in chunk order:
// out = sum_c exp(m_c - M) acc_c / sum_c exp(m_c - M) l_c.
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  pdl_trigger();
  pdl_wait();
  const int seq = blockIdx.x / p.n_head, h = blockIdx.x % p.n_head;
  const int G = p.n_head / p.n_head_kv, kvh = h / G, hl = h - kvh * G;
  const int R = kBlock * G, hd = p.hd, nc = p.n_chunks + 1;
  const size_t slot0 = ((size_t)seq * p.n_head_kv + kvh) * nc;
  for (int e = threadIdx.x; e < kBlock * hd; e += blockDim.x) {
    const int i = e / hd, d = e - i * hd, r = hl * kBlock + i;
    float M = -CUDART_INF_F;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, p.part_ml[((slot0 + c) * R + r) * 2]);
    float L = 0.f, A = 0.f;
    for (int c = 0; c < nc; ++c) {
      const float m = p.part_ml[((slot0 + c) * R + r) * 2];
      if (m == -CUDART_INF_F) continue;
      const float w = expf(m - M);
      L += p.part_ml[((slot0 + c) * R + r) * 2 + 1] * w;
      A += p.part_acc[((slot0 + c) * R + r) * hd + d] * w;
    }
    p.out[(size_t)(seq * kBlock + i) * (p.n_head * hd) + h * hd + d] = A / L;
  }
}

cudaError_t launch_attn_combine(const AttnParams& p, int n_seq, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(n_seq * p.n_head), dim3(128), 0, st, attr);
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
