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

// One CTA = one (sequence, kv head, key chunk).  The G = n_head / n_head_kv
// query heads of the kv group (16 rows each) share the chunk's K/V tile in
// shared memory.  Chunk c < n_chunks covers ring slots [c*chunk, (c+1)*chunk);
// chunk n_chunks is the block's own 16 keys, visible to every row (non-causal).
// A ring slot holding position kp is a key of row i iff 0 <= kp < n_past and
// (n_past + i) - kp < window (dflash-ops model card, Method).  Each CTA writes
// the chunk's row max, sum of exponentials and unnormalised P V.
__global__ void __launch_bounds__(256) attn_chunk_kernel(const __grid_constant__ AttnParams p) {
  const int c = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int G = p.n_head / p.n_head_kv, R = kBlock * G, hd = p.hd;
  const int qd = p.n_head * hd, kvd = p.n_head_kv * hd;
  const bool blk = c == p.n_chunks;
  const int CH = p.chunk < kBlock ? kBlock : p.chunk;
  const int s0 = c * p.chunk;
  const int nk = blk ? kBlock : min(p.chunk, p.window - s0);
  extern __shared__ __align__(16) float sm[];
  float* qT = sm;                 // [hd][R]
  float* kT = qT + hd * R;        // [hd][CH]
  float* vS = kT + hd * CH;       // [CH][hd]
  float* pT = vS + CH * hd;       // [CH][R]
  float* rowm = pT + CH * R;
  float* rowl = rowm + R;
  int* kpos = reinterpret_cast<int*>(rowl + R);
  const int tid = threadIdx.x;
  const int p0 = max(p.n_past[seq], 0);

  for (int idx = tid; idx < R * hd; idx += blockDim.x) {
    const int r = idx / hd, d = idx - r * hd;
    const int hl = r / kBlock, i = r - hl * kBlock;
    qT[d * R + r] = p.q[(size_t)(seq * kBlock + i) * qd + (kvh * G + hl) * hd + d] * p.scale;
  }
  if (blk) {
    for (int idx = tid; idx < kBlock * hd; idx += blockDim.x) {
      const int j = idx / hd, d = idx - j * hd;
      const size_t src = (size_t)(seq * kBlock + j) * kvd + kvh * hd + d;
      kT[d * CH + j] = p.kblk[src];
      vS[j * hd + d] = p.vblk[src];
    }
  } else {
    const size_t plane = (size_t)p.window * hd;
    const size_t kbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 0) * p.n_head_kv + kvh) * plane;
    const size_t vbase = ((((size_t)seq * p.n_layer + p.layer) * 2 + 1) * p.n_head_kv + kvh) * plane;
    for (int idx = tid; idx < nk * hd; idx += blockDim.x) {
      const int j = idx / hd, d = idx - j * hd;
      const size_t o = (size_t)(s0 + j) * hd + d;
      float kv, vv;
      if (p.ring_bf16) {
        const uint16_t* r = reinterpret_cast<const uint16_t*>(p.ring);
        kv = bf16_bits_to_f32(r[kbase + o]);
        vv = bf16_bits_to_f32(r[vbase + o]);
      } else {
        const float* r = reinterpret_cast<const float*>(p.ring);
        kv = r[kbase + o];
        vv = r[vbase + o];
      }
      kT[d * CH + j] = kv;
      vS[j * hd + d] = vv;
    }
    for (int j = tid; j < nk; j += blockDim.x) kpos[j] = p.ring_pos[(size_t)seq * p.window + s0 + j];
  }
  __syncthreads();

  // scores (4 rows x 4 keys per thread), masked, stored transposed [key][row]
  const int nrt = R / 4, nct = (nk + 3) / 4;
  for (int tt = tid; tt < nrt * nct; tt += blockDim.x) {
    const int rt = tt / nct, ct = tt - rt * nct;
    float a[4][4] = {};
    for (int d = 0; d < hd; ++d) {
      const float4 qv = *reinterpret_cast<const float4*>(qT + d * R + 4 * rt);
      const float4 kv = *reinterpret_cast<const float4*>(kT + d * CH + 4 * ct);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w}, ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) a[ii][jj] = fmaf(qa[ii], ka[jj], a[ii][jj]);
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int key = 4 * ct + jj;
      if (key >= nk) continue;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int r = 4 * rt + ii;
        bool ok = true;
        if (!blk) {
          const int kp = kpos[key], qp = p0 + (r % kBlock);
          ok = kp >= 0 && kp < p0 && qp - kp < p.window;
        }
        pT[key * R + r] = ok ? a[ii][jj] : -CUDART_INF_F;
      }
    }
  }
  __syncthreads();
  for (int r = tid; r < R; r += blockDim.x) {
    float m = -CUDART_INF_F;
    for (int key = 0; key < nk; ++key) m = fmaxf(m, pT[key * R + r]);
    float l = 0.f;
    for (int key = 0; key < nk; ++key) {
      const float e = m == -CUDART_INF_F ? 0.f : expf(pT[key * R + r] - m);
      pT[key * R + r] = e;
      l += e;
    }
    rowm[r] = m;
    rowl[r] = l;
  }
  __syncthreads();

  const size_t slot = ((size_t)seq * p.n_head_kv + kvh) * (p.n_chunks + 1) + c;
  float* oacc = p.part_acc + slot * R * hd;
  const int nd8 = hd / 8;
  for (int tt = tid; tt < (R / 4) * nd8; tt += blockDim.x) {
    const int rt = tt / nd8, dt = tt - rt * nd8;
    float o[4][8] = {};
    for (int key = 0; key < nk; ++key) {
      const float4 pv = *reinterpret_cast<const float4*>(pT + key * R + 4 * rt);
      const float4 v0 = *reinterpret_cast<const float4*>(vS + key * hd + 8 * dt);
      const float4 v1 = *reinterpret_cast<const float4*>(vS + key * hd + 8 * dt + 4);
      const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
      const float va[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) o[ii][jj] = fmaf(pa[ii], va[jj], o[ii][jj]);
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      float* dst = oacc + (size_t)(4 * rt + ii) * hd + 8 * dt;
      *reinterpret_cast<float4*>(dst) = make_float4(o[ii][0], o[ii][1], o[ii][2], o[ii][3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(o[ii][4], o[ii][5], o[ii][6], o[ii][7]);
    }
  }
  for (int r = tid; r < R; r += blockDim.x) {
    p.part_ml[(slot * R + r) * 2 + 0] = rowm[r];
    p.part_ml[(slot * R + r) * 2 + 1] = rowl[r];
  }
}

size_t attn_smem_bytes(int group, int hd, int chunk) {
  const int R = kBlock * group, CH = chunk < kBlock ? kBlock : chunk;
  return sizeof(float) * ((size_t)hd * R + (size_t)hd * CH + (size_t)CH * hd + (size_t)CH * R + 2 * R) +
         sizeof(int) * CH;
}

cudaError_t configure_attention(size_t smem) {
  static size_t configured = 0;   // only ever raised, so every live handle still fits
  if (smem <= configured) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) configured = smem;
  return e;
}

cudaError_t launch_attention(const AttnParams& p, int n_seq, cudaStream_t st) {
  const size_t smem = attn_smem_bytes(p.n_head / p.n_head_kv, p.hd, p.chunk);
  dim3 grid(p.n_chunks + 1, p.n_head_kv, n_seq);
  attn_chunk_kernel<<<grid, 256, smem, st>>>(p);
  return cudaGetLastError();
}

// Merge the chunk partials of one (sequence, query head) in chunk order:
// out = sum_c exp(m_c - M) acc_c / sum_c exp(m_c - M) l_c.
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams p) {
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
  attn_combine_kernel<<<n_seq * p.n_head, 128, 0, st>>>(p);
  return cudaGetLastError();
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
