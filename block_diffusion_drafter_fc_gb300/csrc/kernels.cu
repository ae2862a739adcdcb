// Non-GEMM kernels of the drafter step other than attention: block embedding +
// rope tables, the RMSNorm apply of encode, and the first-mismatch acceptance
// scan.
#include "common.cuh"
#include "internal.h"

#include <math_constants.h>

namespace dflash {

// ------------------------------------------------------------------ embedding

// Block rows: token id_last for row 0, mask_token for rows 1..15 (dflash-ops model
// card, Method; dflash_head.rs field mask_token_id).  Writes h (fp32) and the
// row's sums of squares for the first layer's RMSNorm: block b covers part
// b % parts of row b / parts and writes ss[part][row].  Extra blocks (64 entries
// each: fp64 is slow, so it is spread over many SMs) fill the rope table of the
// block positions n_past + i from the host fp64 inverse-frequency table (angle
// and sin/cos in fp64, then rounded to fp32).
__global__ void __launch_bounds__(256) embed_kernel(const void* tok_embd, int dense_bf16, int d,
                                                    int V, int mask_token, const int32_t* id_last,
                                                    const int32_t* n_past, int n_seq,
                                                    const double* inv_freq, int half, float* h,
                                                    float* ss, float2* rope_cs, const void* norm0,
                                                    uint16_t* x_hi, uint16_t* x_lo, int pair_f16,
                                                    int parts, int ss_ld, unsigned* status,
                                                    unsigned long long* stamp) {
  const int M = n_seq * kBlock;
  if (threadIdx.x == 0) stamp_begin(stamp);
  if ((int)blockIdx.x < M * parts) {
    const int m = blockIdx.x / parts, part = blockIdx.x - m * parts, seq = m / kBlock, i = m % kBlock;
    const int span = d / parts, kbeg = part * span, kend = kbeg + span;
    int tok = i == 0 ? id_last[seq] : mask_token;
    if (tok < 0 || tok >= V) {
      if (threadIdx.x == 0 && part == 0) atomicOr(status, 0x1u);
      tok = tok < 0 ? 0 : V - 1;
    }
    // 8 elements per thread and round (one 16-byte bf16 load or two float4
    // loads), all loads of a round issued before any store
    float s = 0.f;
    constexpr int kRound = 4;
    for (int k0 = kbeg + threadIdx.x * 8; k0 < kend; k0 += kRound * (int)blockDim.x * 8) {
      float v[kRound][8];
#pragma unroll
      for (int r = 0; r < kRound; ++r) {
        const int k = k0 + r * blockDim.x * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) v[r][e] = 0.f;
        if (k >= kend) continue;
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
        if (k >= kend) continue;
        float4* dst = reinterpret_cast<float4*>(h + (size_t)m * d + k);
        dst[0] = make_float4(v[r][0], v[r][1], v[r][2], v[r][3]);
        dst[1] = make_float4(v[r][4], v[r][5], v[r][6], v[r][7]);
        // first layer's projection input: h * attn_norm, split into a hi + lo pair
        uint32_t hh[4], ll[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float z0 = v[r][2 * e] * load_dense(norm0, dense_bf16, k + 2 * e);
          const float z1 = v[r][2 * e + 1] * load_dense(norm0, dense_bf16, k + 2 * e + 1);
          split_pair16x2(z0, z1, pair_f16 != 0, hh[e], ll[e]);
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
      ss[(size_t)part * ss_ld + m] = t;
      stamp_finish(stamp);
    }
    return;
  }
  if (threadIdx.x >= 64) return;
  const int e = (blockIdx.x - M * parts) * 64 + threadIdx.x;
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
  if (threadIdx.x == 0) stamp_finish(stamp);
}

cudaError_t launch_embed(const void* tok_embd, int dense_bf16, int n_embd, int n_vocab,
                         int mask_token, const int32_t* id_last, const int32_t* n_past, int n_seq,
                         const double* inv_freq, int hd, float* h, float* ss, float2* rope_cs,
                         const void* norm0, uint16_t* x_hi, uint16_t* x_lo, int pair_f16,
                         int parts, int ss_ld, unsigned* status, unsigned long long* stamp,
                         cudaStream_t st) {
  const int M = n_seq * kBlock, half = hd / 2;
  const int tb = (M * half + 63) / 64;
  if (parts < 1 || n_embd % (8 * parts) != 0) return cudaErrorInvalidValue;
  embed_kernel<<<M * parts + tb, 256, 0, st>>>(tok_embd, dense_bf16, n_embd, n_vocab, mask_token,
                                               id_last, n_past, n_seq, inv_freq, half, h, ss, rope_cs,
                                               norm0, x_hi, x_lo, pair_f16, parts, ss_ld, status,
                                               stamp);
  return cudaGetLastError();
}

// Rope table of injected positions + ring_pos of their slots.  With
// rows_per_seq > 0 the rows belong to consecutive sequences (row t to sequence
// t / rows_per_seq) and, with a count array, only each sequence's first
// count[seq] rows claim their slot.
__global__ void rope_table_kernel(const int32_t* pos, int T, const double* inv_freq, int half,
                                  float2* rope_cs, int32_t* ring_pos, int window, int rows_per_seq,
                                  const int32_t* count, unsigned* status) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= T * half) return;
  const int t = e / half, j = e - t * half;
  int p = pos[t];
  if (p < 0) {
    if (j == 0) atomicOr(status, 0x2u);
    p = 0;
  } else if (j == 0) {
    int sq = 0;
    bool claim = true;
    if (rows_per_seq > 0) {
      sq = t / rows_per_seq;
      claim = !count || t - sq * rows_per_seq < count[sq];
    }
    if (claim) ring_pos[(size_t)sq * window + p % window] = p;
  }
  double sn, cs;
  sincos((double)p * inv_freq[j], &sn, &cs);
  rope_cs[e] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(const int32_t* pos, int T, const double* inv_freq, int hd,
                              float2* rope_cs, int32_t* ring_pos, int window, int rows_per_seq,
                              const int32_t* count, unsigned* status, cudaStream_t st) {
  const int half = hd / 2;
  if (T <= 0) return cudaSuccess;
  rope_table_kernel<<<(T * half + 255) / 256, 256, 0, st>>>(pos, T, inv_freq, half, rope_cs,
                                                            ring_pos, window, rows_per_seq, count,
                                                            status);
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

// ------------------------------------------------------------------ acceptance

// One warp per sequence: lanes 0..14 compare draft j with the target's token j,
// a ballot marks the mismatches, and the first set bit is the number of leading
// matches (15 when none): dflash-ops model card, Usage (device-side accept) and
// dflash_engine.py, DFlashSpeculativeVerifier.verify_block.
__global__ void accept_kernel(const int32_t* drafts, const int32_t* targets, int32_t* n_ok,
                              int n_seq, int width, unsigned long long* stamp) {
  const int seq = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) stamp_begin(stamp);
  if (seq >= n_seq) return;
  bool miss = false;
  if (lane < kBlock - 1)
    miss = lane >= width - 1 || drafts[seq * (kBlock - 1) + lane] != targets[seq * (kBlock - 1) + lane];
  const unsigned mask = __ballot_sync(0xffffffffu, miss);
  if (lane == 0) n_ok[seq] = mask ? __ffs(mask) - 1 : kBlock - 1;
  if (threadIdx.x == 0) stamp_finish(stamp);
}

cudaError_t launch_accept(const int32_t* drafts, const int32_t* targets, int32_t* n_ok, int n_seq,
                          int width, unsigned long long* stamp, cudaStream_t st) {
  accept_kernel<<<(n_seq + 7) / 8, 256, 0, st>>>(drafts, targets, n_ok, n_seq, width, stamp);
  return cudaGetLastError();
}

// One turn of the speculative loop after the target's verification, one warp
// per sequence (dflash_engine.py, DFlashSpeculativeVerifier.verify_block;
// dflash-ops model card, Usage): m = number of leading drafts equal to the
// target's tokens; the accepted block rows 0..m (positions n_past .. n_past + m)
// are the rows to inject, the target's token m becomes the next id_last, and
// n_past advances by m + 1.  Writes pos[16 s + i] = n_past + i for all 16 rows
// and count[s] = m + 1.
__global__ void advance_kernel(const int32_t* drafts, const int32_t* targets, int n_seq, int width,
                               int32_t* id_last, int32_t* n_past, int32_t* n_ok, int32_t* pos,
                               int32_t* count) {
  const int seq = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (seq >= n_seq) return;
  bool miss = false;
  if (lane < kBlock - 1)
    miss = lane >= width - 1 || drafts[seq * (kBlock - 1) + lane] != targets[seq * kBlock + lane];
  const unsigned mask = __ballot_sync(0xffffffffu, miss);
  const int m = mask ? __ffs(mask) - 1 : kBlock - 1;
  const int p0 = n_past[seq];
  __syncwarp();
  if (lane < kBlock) pos[seq * kBlock + lane] = p0 + lane;
  if (lane == 0) {
    n_ok[seq] = m;
    count[seq] = m + 1;
    id_last[seq] = targets[seq * kBlock + m];
    n_past[seq] = p0 + m + 1;
  }
}

cudaError_t launch_advance(const int32_t* drafts, const int32_t* targets, int n_seq, int width,
                           int32_t* id_last, int32_t* n_past, int32_t* n_ok, int32_t* pos,
                           int32_t* count, cudaStream_t st) {
  advance_kernel<<<(n_seq + 7) / 8, 256, 0, st>>>(drafts, targets, n_seq, width, id_last, n_past,
                                                  n_ok, pos, count);
  return cudaGetLastError();
}

// fp32 rows -> the hi / lo pair a projection reads (bf16, or fp16 with FP4
// weights; two values per thread)
__global__ void split_pair_kernel(const float* x, int n, uint16_t* hi, uint16_t* lo, int pair_f16) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float2 v = i + 1 < n ? *reinterpret_cast<const float2*>(x + i) : make_float2(x[i], 0.f);
  uint32_t h, l;
  split_pair16x2(v.x, v.y, pair_f16 != 0, h, l);
  if (i + 1 < n) {
    *reinterpret_cast<uint32_t*>(hi + i) = h;
    *reinterpret_cast<uint32_t*>(lo + i) = l;
  } else {
    hi[i] = (uint16_t)(h & 0xffffu);
    lo[i] = (uint16_t)(l & 0xffffu);
  }
}

cudaError_t launch_split_pair(const float* x, int n, uint16_t* hi, uint16_t* lo, int pair_f16,
                              cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int pairs = (n + 1) / 2;
  split_pair_kernel<<<(pairs + 255) / 256, 256, 0, st>>>(x, n, hi, lo, pair_f16);
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
