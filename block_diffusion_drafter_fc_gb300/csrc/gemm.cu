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
#include "gemm_common.cuh"

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

// Four consecutive norm weights as fp32 (vector load of the dense dtype).
DF_DEVICE float4 load_norm4(const void* w, int bf16, int k) {
  if (bf16) {
    const uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(w) + k);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
  }
  return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(w) + k);
}

// Activation rows m0..m0+15, columns [xs0, xs0+xlen) -> bf16 hi/lo in shared
// memory.  Each thread first issues all of its loads (up to kStageVec groups of
// four elements), then normalises, splits and stores, so one stage costs about
// one L2 round trip.
constexpr int kStageVec = 4;

DF_DEVICE void stage_x(const GemmParams& p, uint16_t* xh, uint16_t* xl, int XS,
                       const float* inv_rms, int m0, int xs0, int xlen) {
  const int q4 = xlen >> 2, total = 16 * q4;
  for (int base = 0; base < total; base += kStageVec * kGemmThreads) {
    float4 v[kStageVec];
    float4 w[kStageVec];
#pragma unroll
    for (int u = 0; u < kStageVec; ++u) {
      const int idx = base + u * kGemmThreads + threadIdx.x;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      w[u] = make_float4(1.f, 1.f, 1.f, 1.f);
      if (idx < total) {
        const int m = idx / q4, c = (idx - m * q4) * 4;
        const int row = m0 + m, k = xs0 + c;
        if (row < p.M) {
          if (p.x_mode == X_BF16) {
            const uint2 b = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.x) +
                                                            (size_t)row * p.ldx + k);
            v[u] = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u),
                               __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u));
          } else {
            v[u] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.x) +
                                                    (size_t)row * p.ldx + k);
          }
        }
        if (p.normw) w[u] = load_norm4(p.normw, p.norm_bf16, k);
      }
    }
#pragma unroll
    for (int u = 0; u < kStageVec; ++u) {
      const int idx = base + u * kGemmThreads + threadIdx.x;
      if (idx >= total) continue;
      const int m = idx / q4, c = (idx - m * q4) * 4;
      float4 f = v[u];
      if (p.normw) {
        const float r = inv_rms[m];
        f.x = f.x * r * w[u].x;
        f.y = f.y * r * w[u].y;
        f.z = f.z * r * w[u].z;
        f.w = f.w * r * w[u].w;
      }
      uint2 hi, lo;
      split_bf16x2(f.x, f.y, hi.x, lo.x);
      split_bf16x2(f.z, f.w, hi.y, lo.y);
      *reinterpret_cast<uint2*>(xh + m * XS + c) = hi;
      *reinterpret_cast<uint2*>(xl + m * XS + c) = lo;
    }
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

// ------------------------------------------------------------------ kernel

template <int WT>
__global__ void __launch_bounds__(kGemmThreads, 2) gemm_rows_kernel(const __grid_constant__ GemmParams p) {
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
      // weights do not depend on the activations: pull this stage's rows into L2
      // and start the register pipeline before staging x (and, for the first
      // stage, before waiting for the previous kernel)
      if (lane < 16) {
        const uint8_t* row = map_row(p, tile, warp * 16 + lane, T::ESZ, &dummy);
        if (row) prefetch_l2(row + (size_t)xs0 * T::ESZ, (uint32_t)(xlen * T::ESZ));
      }
      load_stage<WT>(ra, rb, pa, pb, 0, nch);
      if (!waited) {
        pdl_wait();  // everything below may read what earlier kernels wrote
        waited = true;
      }
      if (xs0 == k0 && p.normw) compute_inv_rms(p, inv_rms, m0);
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

    if (!segment_fixup(p, acc_s, item, c0, c1, U, G, b, &s_flag)) continue;
    run_epilogue(p, acc_s, scale_s, inv_rms, mb, tile, &s_flag);
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
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
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
