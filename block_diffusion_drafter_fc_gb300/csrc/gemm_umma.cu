// Dense projection kernel on the 5th-generation tensor cores (tcgen05), for
// steps with at least 128 activation rows (the cross-sequence batch of
// dflash_head.rs, struct DflashBatch: 16 rows per sequence).
//
// Persistent: one CTA per SM walks output tiles D[128 activation rows][128
// weight rows] (tile t = CTA, CTA + grid, ...; consecutive tiles share a weight
// tile across the activation row blocks, so weights come from HBM once), each
// over the whole k range, with the accumulator double-buffered in tensor memory
// so that a tile's epilogue overlaps the next tile's MMAs:
//   warp 12 (one lane)  TMA producer: per 64-wide k chunk, the activation hi and
//                       lo boxes [128 rows x 128 B] and the weight box(es) into
//                       a 3-stage shared-memory ring (128-byte swizzle, the UMMA
//                       K-major canonical layout), across tile boundaries;
//   warps 8..11         E4M3 weights only: widen the raw [128 x 64] byte tile to
//                       the bf16 swizzled tile the MMA reads (exact), then fence
//                       the generic-proxy writes for the async proxy;
//   warp 13 (one lane)  allocates 2 x 128 TMEM columns and issues, per k16 step,
//                       tcgen05.mma kind::f16 (bf16 x bf16, fp32 accumulate) for
//                       the activation hi part and again for the lo part (the
//                       fp32 activations are split into bf16 hi + lo) into the
//                       tile's accumulator buffer; commits each stage back to
//                       the producer and each finished tile to the epilogue;
//   warps 0..7          per 32-lane quadrant of the accumulator, tcgen05.ld into
//                       two 16-row blocks in shared memory and the fused
//                       epilogues of the 16-row kernels on each (RMS row scale,
//                       per-head q/k norm + rope, residual + next input, SwiGLU,
//                       logits + argmax); then hand the buffer back to the MMA.
// Every mbarrier wait gives up after ~2 s with DFLASH_DEV_TIMEOUT; tensor memory
// is always released before exit.
#include "gemm_common.cuh"

namespace dflash {

namespace umma {

constexpr int kS = 3;                  // pipeline stages
constexpr int kTile = 128 * 128;       // bytes of one [128 rows x 128 B] swizzled tile
constexpr long long kWait = 4000000000LL;
constexpr int kThreads = 448;          // warps 0-7 epilogue, 8-11 E4M3 widening, 12 TMA, 13 MMA
constexpr int kWiden = 4;              // widening warps
constexpr int kBRow = kTileRows + 4;   // padded row (floats) of a read-out block

// Shared-memory layout for output tiles of 128 activation rows x WR weight rows
// (WR = 128, or 256 = two 128-row n-tiles sharing every activation chunk).
template <int WR>
struct L {
  static constexpr int kWTile = WR * 128;   // bf16 [WR x 64] swizzled weight tile
  static constexpr int kWRaw = WR * 64;     // raw [WR x 64] E4M3 (upper half of kWTile)
  static constexpr int kAccCols = WR;       // TMEM columns of one accumulator buffer (fp32)
  // stage: A hi | A lo | B (bf16; E4M3 lands raw in its upper half, widened in place)
  static constexpr int kStage = 2 * kTile + kWTile;
  static constexpr int kOffBlk = kS * kStage;                  // two 16-row read-out blocks
  static constexpr int kOffAcc = kOffBlk + 2 * 16 * kBRow * 4; // one 16 x 128 fp32 epilogue tile
  static constexpr int kOffInv = kOffAcc + 16 * kTileRows * 4;
  static constexpr int kOffScale = kOffInv + 16 * 4;
  static constexpr int kOffBars = kOffScale + kTileRows * 4;   // full, conv, empty [S], accf, acce [2]
  static constexpr int kOffTmem = kOffBars + (3 * kS + 4) * 8;
  static constexpr int kSmem = kOffTmem + 16 + 1024;           // + alignment slack
  static_assert(kSmem <= 227 * 1024, "shared memory of the tcgen05 projection");
};

DF_DEVICE uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

DF_DEVICE void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
DF_DEVICE void bar_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
DF_DEVICE void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
DF_DEVICE bool bar_try(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(par)
      : "memory");
  return ok != 0;
}
DF_DEVICE bool bar_wait(uint64_t* b, uint32_t par) {
  if (bar_try(b, par)) return true;
  const long long t0 = clock64();
  while (!bar_try(b, par))
    if (clock64() - t0 > kWait) return false;
  return true;
}

DF_DEVICE void tma2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(su32(b))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes in 8-row (1024-byte) groups.
DF_DEVICE uint64_t desc_sw128(const void* p) {
  const uint64_t a = su32(p);
  return ((a >> 4) & 0x3FFFull) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major, M x N.
constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

DF_DEVICE void mma_f16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
DF_DEVICE void mma_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   su32(b))
               : "memory");
}

}  // namespace umma

template <int WT, int WR>
__global__ void __launch_bounds__(umma::kThreads, 1) gemm_umma_kernel(const __grid_constant__ GemmParams p) {
  using namespace umma;
  using Lt = L<WR>;
  constexpr int kWTile = Lt::kWTile, kWRaw = Lt::kWRaw, kAccCols = Lt::kAccCols, kStage = Lt::kStage;
  constexpr int kOffBlk = Lt::kOffBlk, kOffAcc = Lt::kOffAcc, kOffInv = Lt::kOffInv;
  constexpr int kOffScale = Lt::kOffScale, kOffBars = Lt::kOffBars, kOffTmem = Lt::kOffTmem;
  constexpr int kNsub = WR / 128;   // 128-row n-tiles per output tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* blk = reinterpret_cast<float*>(sm + kOffBlk);
  float* acc_s = reinterpret_cast<float*>(sm + kOffAcc);
  float* inv_rms = reinterpret_cast<float*>(sm + kOffInv);
  float* scale_s = reinterpret_cast<float*>(sm + kOffScale);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOffBars);
  uint64_t* conv = full + kS;
  uint64_t* empty = conv + kS;
  uint64_t* accf = empty + kS;   // accumulator buffer b holds a finished tile
  uint64_t* acce = accf + 2;     // accumulator buffer b has been read out
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmem);
  __shared__ int s_flag;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool fp8 = WT == W_FP8;
  const int m_tiles = (p.M + 127) / 128;
  const int n_items = m_tiles * ((p.n_tiles + kNsub - 1) / kNsub);   // 128 act rows x WR weight rows
  const int nk = p.cpt;                            // 64-wide k chunks
  const int G = gridDim.x;
  if (tid == 0) {
    for (int s = 0; s < kS; ++s) {
      bar_init(&full[s], 1);
      bar_init(&conv[s], kWiden);
      bar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      bar_init(&accf[b], 1);
      bar_init(&acce[b], 8);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    stamp_begin(p.stamp);
  }
  if (warp == 13) {  // two accumulator buffers of WR fp32 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_slot)), "n"(2 * WR)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 12) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      pdl_wait();
      const uint32_t bytes = kTile * (p.has_lo ? 2 : 1) + (fp8 ? kWRaw : kWTile);
      long long it = 0;
      for (int t = blockIdx.x; t < n_items && !s_abort; t += G) {
        const int mt = t % m_tiles, wt2 = t / m_tiles;
        int maps[WR / 32], rows[WR / 32];
#pragma unroll
        for (int q = 0; q < WR / 32; ++q) {  // the WR weight rows in 32-row boxes, per segment map
          const int nt = kNsub * wt2 + (q >> 2), qq = q & 3;
          if (p.map == MAP_SWIGLU) {
            maps[q] = qq < 2 ? 0 : 1;
            rows[q] = nt * (kTileRows / 2) + (qq & 1) * 32;
          } else {
            const int vr = nt * kTileRows + qq * 32;   // past N: read as zeros
            int s = 0;
            while (s + 1 < p.nseg && vr >= p.seg[s + 1].row0) ++s;
            maps[q] = s;
            rows[q] = vr - p.seg[s].row0;
          }
        }
        for (int k = 0; k < nk; ++k, ++it) {
          const int st = (int)(it % kS);
          if (!bar_wait(&empty[st], (uint32_t)((it / kS) & 1) ^ 1)) {
            atomicOr(p.status, 0x4u);
            s_abort = 1;
            break;
          }
          uint8_t* base = sm + st * kStage;
          bar_expect(&full[st], bytes);
          tma2d(base, &p.tm_xh, k * 64, mt * 128, &full[st]);
          if (p.has_lo) tma2d(base + kTile, &p.tm_xl, k * 64, mt * 128, &full[st]);
          uint8_t* bdst = fp8 ? base + 2 * kTile + kWRaw : base + 2 * kTile;
          const int box_bytes = fp8 ? 32 * 64 : 32 * 128;
#pragma unroll
          for (int q = 0; q < WR / 32; ++q) tma2d(bdst + q * box_bytes, &p.tm_w[maps[q]], k * 64, rows[q], &full[st]);
        }
      }
      // no copy may still be landing when the CTA exits
      for (long long j = it > kS ? it - kS : 0; j < it; ++j)
        if (!bar_wait(&full[j % kS], (uint32_t)((j / kS) & 1))) {
          atomicOr(p.status, 0x4u);
          break;
        }
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, WR);
      long long it = 0;
      int i = 0;
      for (int t = blockIdx.x; t < n_items && !s_abort; t += G, ++i) {
        const int buf = i & 1;
        if (!bar_wait(&acce[buf], (uint32_t)((i >> 1) & 1) ^ 1)) {  // epilogue done with it
          atomicOr(p.status, 0x4u);
          s_abort = 1;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t acc = tmem + buf * kAccCols;
        for (int k = 0; k < nk; ++k, ++it) {
          const int st = (int)(it % kS);
          uint64_t* ready = fp8 ? &conv[st] : &full[st];
          if (!bar_wait(ready, (uint32_t)((it / kS) & 1))) {
            atomicOr(p.status, 0x4u);
            s_abort = 1;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          uint8_t* base = sm + st * kStage;
          const uint64_t da = desc_sw128(base), dl = desc_sw128(base + kTile),
                         db = desc_sw128(base + 2 * kTile);
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // 16 k per MMA: +32 bytes inside the swizzled rows
            const uint64_t adv = (uint64_t)(j * 32) >> 4;
            mma_f16(acc, da + adv, db + adv, idesc, (k | j) != 0);
            if (p.has_lo) mma_f16(acc, dl + adv, db + adv, idesc, 1);
          }
          mma_commit(&empty[st]);
        }
        mma_commit(&accf[buf]);
      }
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------------- E4M3 widening
    if (fp8) {
      const int wt = tid - 256;  // 0..127
      long long it = 0;
      for (int t = blockIdx.x; t < n_items; t += G) {
        for (int k = 0; k < nk; ++k, ++it) {
          const int st = (int)(it % kS);
          if (!s_abort && !bar_wait(&full[st], (uint32_t)((it / kS) & 1))) {
            if (lane == 0) atomicOr(p.status, 0x4u);
            s_abort = 1;
          }
          uint8_t* base = sm + st * kStage;
          uint8_t* dst = base + 2 * kTile;          // [WR rows][128 B] bf16, 128-byte swizzle
          const uint8_t* raw = dst + kWRaw;         // [WR rows][64 B] E4M3, unswizzled
          // WR rows x 4 (16-byte raw pieces) over 128 threads: all read before any
          // write (the raw bytes sit in the widened tile's upper half)
          uint4 v[WR / 32];
#pragma unroll
          for (int u = 0; u < WR / 32; ++u) {
            const int pc = wt + u * 128;
            v[u] = *reinterpret_cast<const uint4*>(raw + (pc >> 2) * 64 + (pc & 3) * 16);
          }
          asm volatile("bar.sync 2, %0;" ::"n"(32 * kWiden) : "memory");
#pragma unroll
          for (int u = 0; u < WR / 32; ++u) {
            const int pc = wt + u * 128;
            const int row = pc >> 2, q = pc & 3;
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              o[2 * e] = e4m3x2_to_bf16x2((uint16_t)(w[e] & 0xffffu));
              o[2 * e + 1] = e4m3x2_to_bf16x2((uint16_t)(w[e] >> 16));
            }
            // 16 E4M3 = 32 bf16 bytes = chunks 2q and 2q + 1 of the bf16 row
            *reinterpret_cast<uint4*>(dst + row * 128 + (((2 * q) ^ (row & 7)) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + row * 128 + (((2 * q + 1) ^ (row & 7)) << 4)) =
                make_uint4(o[4], o[5], o[6], o[7]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          // every widening warp is done reading this stage's raw bytes before the
          // next use of the buffer can be refilled (it follows the MMA's commit)
          __syncwarp();
          if (lane == 0) bar_arrive(&conv[st]);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue warps 0..7
    pdl_wait();
    const int quad = warp & 3, half = warp >> 2;
    int i = 0;
    for (int t = blockIdx.x; t < n_items; t += G, ++i) {
      const int mt = t % m_tiles, wt2 = t / m_tiles;
      const int buf = i & 1;
      const bool ok = s_abort || bar_wait(&accf[buf], (uint32_t)((i >> 1) & 1));
      if (!ok && lane == 0) atomicOr(p.status, 0x4u);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      for (int sub = 0; sub < kNsub; ++sub) {
        const int nt = kNsub * wt2 + sub;
        if (nt >= p.n_tiles) break;
        csync();  // the previous n-tile's epilogues are done with scale_s
        if (tid < kTileRows) {  // scales of this n-tile's weight rows
          const float* sc = nullptr;
          const uint8_t* r = map_row(p, nt, tid, 1, &sc);
          scale_s[tid] = r ? (sc ? *sc : 1.f) : 0.f;
        }
        for (int q = 0; q < 4; ++q) {
          const int mb0 = mt * 8 + 2 * q;    // the quadrant's two 16-row blocks
          if (mb0 * 16 >= p.M) break;
          if (quad == q) {
            // lanes 32q..32q+31 of the accumulator, this warp's half of the
            // n-tile's columns, into block (lane / 16) row (lane % 16) (padded
            // rows: the 32 lanes' rows do not share banks)
            float* row = blk + (size_t)(lane >> 4) * 16 * kBRow + (size_t)(lane & 15) * kBRow;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t r[32];
              const uint32_t taddr = tmem + buf * kAccCols + ((uint32_t)(q * 32) << 16) + sub * 128 +
                                     half * 64 + c * 32;
              asm volatile(
                  "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
                  "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                  : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                    "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                    "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
                    "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
                    "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
                    "=r"(r[31])
                  : "r"(taddr));
              asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(row + half * 64 + c * 32 + e) =
                    make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
            }
          }
          csync();
          for (int b2 = 0; b2 < 2; ++b2) {
            const int mb = mb0 + b2;
            if (mb * 16 >= p.M) break;
            for (int e = tid; e < 16 * kTileRows; e += kGemmThreads) {
              const int m = e / kTileRows, c = e - m * kTileRows;
              acc_s[e] = blk[(size_t)(b2 * 16 + m) * kBRow + c];
            }
            if (p.row_scale) compute_inv_rms(p, inv_rms, mb * 16);
            csync();
            run_epilogue(p, acc_s, scale_s, inv_rms, mb, nt, &s_flag);
            csync();
          }
        }
      }
      // the accumulator buffer may be overwritten by the next tile's MMAs
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) bar_arrive(&acce[buf]);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0) stamp_finish(p.stamp);
  if (warp == 13) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(2 * WR) : "memory");
  }
}

size_t gemm_umma_smem_bytes() { return umma::L<256>::kSmem; }

cudaError_t configure_gemm_umma() {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* fn, int bytes) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  };
  set(reinterpret_cast<const void*>(gemm_umma_kernel<W_BF16, 128>), umma::L<128>::kSmem);
  set(reinterpret_cast<const void*>(gemm_umma_kernel<W_BF16, 256>), umma::L<256>::kSmem);
  set(reinterpret_cast<const void*>(gemm_umma_kernel<W_FP8, 128>), umma::L<128>::kSmem);
  set(reinterpret_cast<const void*>(gemm_umma_kernel<W_FP8, 256>), umma::L<256>::kSmem);
  return e;
}

template <int WT, int WR>
static cudaError_t launch_umma_t(const GemmParams& p, int n_sm, cudaStream_t st) {
  const int items = (p.M + 127) / 128 * ((p.n_tiles + WR / 128 - 1) / (WR / 128));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items < n_sm ? items : n_sm);   // persistent: one CTA per SM
  cfg.blockDim = dim3(umma::kThreads);
  cfg.dynamicSmemBytes = umma::L<WR>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_umma_kernel<WT, WR>, p);
}

// 256-row weight tiles (half the activation traffic per flop) when they still
// give every SM a tile, else 128-row tiles for more parallelism.  The logits
// epilogue (an fp32 store of every output plus the argmax partials) is the
// heaviest; its tiles stay 128 rows so that it keeps pace with the MMAs.
cudaError_t launch_gemm_umma(int wt, const GemmParams& p, cudaStream_t st) {
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (n_sm <= 0) n_sm = 1;
  }
  const bool wide = p.epi != EPI_LOGITS && (p.M + 127) / 128 * ((p.n_tiles + 1) / 2) >= n_sm;
  if (wt == W_BF16) return wide ? launch_umma_t<W_BF16, 256>(p, n_sm, st) : launch_umma_t<W_BF16, 128>(p, n_sm, st);
  if (wt == W_FP8) return wide ? launch_umma_t<W_FP8, 256>(p, n_sm, st) : launch_umma_t<W_FP8, 128>(p, n_sm, st);
  return cudaErrorInvalidValue;
}

}  // namespace dflash
