// Projection kernel for FP4 weights on the 5th-generation tensor cores.
//
// y[m][n] = s[n] sum_k x[m][k] w[n][k] for 16-row activation blocks, with w the
// FP4 weights of include/dflash.h (E2M1 codes, an E4M3 scale per 16 weights of
// a row).  At 16 activation rows the weights are a 4.5-bit stream that the
// 16-row mma.sync kernel cannot keep up with (its fp16 products, doubled by the
// hi/lo split of the activations, saturate the warp-level tensor path before
// HBM does).  Here the decoded weights never touch shared memory: they go to
// tensor memory as the A operand of tcgen05.mma (M = 128 weight rows, K = 16),
// and the activation pair stays in shared memory as B: its 16 hi rows and 16 lo
// rows are one N = 32 operand, and the epilogue adds the two halves of the
// accumulator.
//
// Stream-K over 128-row x 256-k units as in the 16-row kernels (one CTA per
// SM, each a contiguous run of units; shared tiles summed by the last
// contributor in CTA order), warp-specialised:
//   warp 16 (one lane) TMA producer: per unit the tile's codes (a 64-row box of
//                      128 bytes per row for every four 16-row groups of one
//                      segment, else 16-row boxes), their block scales (a
//                      2-D box of 4 groups x 256 bytes, else 256 contiguous
//                      bytes per group) and the activation pair (per 64 k a
//                      16-row hi box followed by its lo box: one 32-row
//                      operand; one 4-D copy, else 8 boxes) into a 5-stage
//                      ring, across tile boundaries;
//   warps 8..15        decoders: warp w owns TMEM lanes 32 (w % 4) .. + 31 (the
//                      tile's rows) and half of the unit's k; a lane widens its
//                      row's 128 codes with cvt.rn.f16x2.e2m1x2, multiplies
//                      them by their block scale in fp16 (exact: at most six
//                      significant bits, within [2^-10, 2688]) and stores the 64
//                      fp16 pairs with tcgen05.st into one of two A buffers;
//   warps 0..7         at the end of each segment read the accumulator
//                      (tcgen05.ld) into the 16 x 128 tile of the shared fix-up
//                      and run the fused epilogue, while the decoders and MMA
//                      warps go on with the next segment;
//   warps 17..20       (one lane each) per unit 4 k-step MMAs each into its own
//                      accumulator of the segment (one of two per warp; the
//                      epilogue adds the eight halves: a single issuing thread
//                      cannot keep up with 16 MMAs per 18 KB), committing the stage
//                      back to the producer and the A buffer back to the
//                      decoders; warp 17 allocates tensor memory.
// Every mbarrier wait gives up after ~2 s with DFLASH_DEV_TIMEOUT and the CTA
// runs to its end without further waits; tensor memory is always released.
#include "gemm_common.cuh"

namespace dflash {

namespace fp4 {

constexpr int kBox = 16 * 128;              // one 16-row x 128-byte box
constexpr int kScaleBox = 256;              // block scales of 16 rows x 256 k
constexpr int kX = 4 * kBox;                // 256 k of one half of the activation pair
constexpr int kAB = 2;                      // A buffers (128 TMEM columns each)
constexpr int kDB = 2;                      // accumulator buffers per MMA warp (32 columns each)
// Shared-memory layout per weight format: a unit's codes (FP4: 128 bytes per
// row and its block scales; E4M3: two 128-byte k halves per row), the
// activation pair, and the fix-up / epilogue area
template <int WF>
struct Lay {
  static constexpr int kS = WF == W_FP8 ? 4 : 5;                      // pipeline stages
  static constexpr int kCodes = (WF == W_FP8 ? 2 : 1) * 8 * kBox;     // the tile's code boxes
  static constexpr int kScales = WF == W_FP8 ? 0 : 8 * kScaleBox;
  static constexpr int kStage = kCodes + kScales + 2 * kX;
  static constexpr int kOffAcc = kS * kStage;        // 16 x 128 fp32 fix-up tile
  static constexpr int kOffInv = kOffAcc + 16 * kTileRows * 4;
  static constexpr int kOffScale = kOffInv + 16 * 4;
  static constexpr int kOffBars = kOffScale + kTileRows * 4;   // full, empty [S]; afull, aempty [AB]; accf, acce [DB]
  static constexpr int kOffTmem = kOffBars + (2 * kS + 2 * kAB + 2 * kDB) * 8;
  static constexpr int kSmem = kOffTmem + 16 + 1024;            // + alignment slack
  static_assert(kStage % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled boxes");
  static_assert(kSmem <= 227 * 1024 && kSmem > 114 * 1024, "one CTA per SM (it owns the SM's TMEM)");
};
constexpr int kEpilogue = 8;                // warps 0..7: segment read-out, fix-up and epilogue
constexpr int kDecoders = 8;                // warps 8..15: decoding
constexpr int kIssuers = 4;                 // MMA warps: issuer i takes k16 steps 4i .. 4i + 3
constexpr int kThreads = 32 * (kEpilogue + kDecoders + 1 + kIssuers);
constexpr int kProducer = kEpilogue + kDecoders, kIssuer = kProducer + 1;
constexpr int kTmemCols = 512;              // A: 2 x 128 columns; D: issuers x 2 x 32 columns
constexpr int kDCol = 128 * kAB;
static_assert(kDCol + kIssuers * kDB * 32 <= kTmemCols, "tensor memory columns");
constexpr long long kWait = 4000000000LL;

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
DF_DEVICE void tma4d(void* dst, const CUtensorMap* map, int x0, int x1, int x2, int x3, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(su32(dst)),
      "l"(map), "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(su32(b))
      : "memory");
}
DF_DEVICE void tma2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* b, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(su32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(su32(b)), "l"(pol)
      : "memory");
}
DF_DEVICE void bulk_hint(void* dst, const void* src, uint32_t bytes, uint64_t* b, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(b)), "l"(pol)
      : "memory");
}
DF_DEVICE uint64_t evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// K-major operand in shared memory, 128-byte swizzle, 8-row groups of 1024 bytes.
DF_DEVICE uint64_t desc_sw128(uint32_t a) {
  return ((uint64_t)(a >> 4) & 0x3FFFull) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}
// kind::f16 with fp16 A and B, fp32 D, K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D (tmem) += A (tmem) x B (shared memory descriptor)
DF_DEVICE void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
DF_DEVICE void commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   su32(b))
               : "memory");
}

// The eight E2M1 codes of a word as four fp16x2 (byte j -> element j; low
// nibble -> low half): exact.
DF_DEVICE void e2m1x8(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}
// An E4M3 scale as an fp16 pair {s, s}.
DF_DEVICE uint32_t e4m3_pair(uint32_t b) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(b * 0x101u), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
DF_DEVICE uint32_t hmul2u(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 32 consecutive TMEM columns of this warp's 32 lanes <- 32 registers per thread
DF_DEVICE void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]));
}

// byte offset of (row, 16-byte chunk) inside a 128-byte-swizzled box
DF_DEVICE int swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

// Tensor-map index and row coordinate of 16-row group `grp` of `tile`
DF_DEVICE void group_coord(const GemmParams& p, int tile, int grp, int& map, int& row) {
  if (p.map == MAP_SWIGLU) {
    map = grp < 4 ? 0 : 1;
    row = tile * (kTileRows / 2) + (grp & 3) * 16;
    return;
  }
  const int vr = tile * kTileRows + grp * 16;
  int s = 0;
  while (s + 1 < p.nseg && vr >= p.seg[s + 1].row0) ++s;
  map = s;
  row = vr - p.seg[s].row0;
}

// This CTA's 1/G share of the L2 prefetch ranges of the next kernel's input.
DF_DEVICE void prefetch_share(const GemmParams& p, int b, int G) {
  const unsigned long long total = p.pf_bytes * (unsigned long long)p.pf_count;
  const unsigned long long x0 = (total * b / G) & ~15ull;
  const unsigned long long x1 = b == G - 1 ? total : (total * (b + 1) / G) & ~15ull;
  for (unsigned long long x = x0; x < x1;) {
    const unsigned long long i = x / p.pf_bytes, off = x - i * p.pf_bytes;
    unsigned long long n = p.pf_bytes - off;
    if (n > x1 - x) n = x1 - x;
    if (n > 32768) n = 32768;
    prefetch_l2(p.pf_base + i * p.pf_stride + off, (uint32_t)n);
    x += n;
  }
}

}  // namespace fp4

template <int WF>
__global__ void __launch_bounds__(fp4::kThreads, 1) gemm_fp4_kernel(const __grid_constant__ GemmParams p) {
  using namespace fp4;
  using Lt = Lay<WF>;
  constexpr int kS = Lt::kS, kStage = Lt::kStage, kCodes = Lt::kCodes, kScales = Lt::kScales;
  constexpr int kOffAcc = Lt::kOffAcc, kOffInv = Lt::kOffInv, kOffScale = Lt::kOffScale;
  constexpr int kOffBars = Lt::kOffBars, kOffTmem = Lt::kOffTmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* acc_s = reinterpret_cast<float*>(sm + kOffAcc);
  float* inv_rms = reinterpret_cast<float*>(sm + kOffInv);
  float* scale_s = reinterpret_cast<float*>(sm + kOffScale);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOffBars);
  uint64_t* empty = full + kS;
  uint64_t* afull = empty + kS;   // A buffer a decoded
  uint64_t* aempty = afull + kAB; // A buffer a read by its MMAs
  uint64_t* accf = aempty + kAB;  // accumulator d holds a finished segment
  uint64_t* acce = accf + kDB;    // accumulator d has been read out
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmem);
  __shared__ int s_flag;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kS; ++s) {
      bar_init(&full[s], 1);
      bar_init(&empty[s], kIssuers);
    }
    for (int a = 0; a < kAB; ++a) {
      bar_init(&afull[a], kDecoders);
      bar_init(&aempty[a], kIssuers);
    }
    for (int b = 0; b < kDB; ++b) {
      bar_init(&accf[b], kIssuers);
      bar_init(&acce[b], kEpilogue);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    stamp_begin(p.stamp);
  }
  if (warp == kIssuer) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_slot)), "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  const int G = gridDim.x, b = blockIdx.x;
  const long long U = (long long)p.n_tiles * p.n_mb * p.cpt;
  const long long ub0 = U * b / G, ub1 = U * (b + 1) / G;

  if (warp == kProducer) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = evict_first();
      long long it = 0;
      bool waited = false;
      for (long long u = ub0; u < ub1 && !s_abort;) {
        const int item = (int)(u / p.cpt);
        const int c0 = (int)(u - (long long)item * p.cpt);
        const int c1 = (int)min((long long)p.cpt, c0 + (ub1 - u));
        u += c1 - c0;
        const int tile = item / p.n_mb, mb = item - tile * p.n_mb;
        int gmap[8], grow[8];
#pragma unroll
        for (int grp = 0; grp < 8; ++grp) group_coord(p, tile, grp, gmap[grp], grow[grp]);
        for (int c = c0; c < c1; ++c, ++it) {
          const int st = (int)(it % kS);
          if (!bar_wait(&empty[st], (uint32_t)((it / kS) & 1) ^ 1)) {
            atomicOr(p.status, 0x4u);
            s_abort = 1;
            break;
          }
          uint8_t* dst = sm + st * kStage;
          bar_expect(&full[st], kStage);
#pragma unroll
          for (int hq = 0; hq < 2 && WF == W_FP8; ++hq) {
            // E4M3: the unit's 256 k of each row are two 128-byte halves
            const int g0 = 4 * hq;
            const bool w64 = p.w64 && gmap[g0 + 3] == gmap[g0] && grow[g0 + 3] == grow[g0] + 48;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
              uint8_t* cd = dst + kb * (8 * kBox);
              if (w64) {
                tma2d_hint(cd + g0 * kBox, &p.tm_w64[gmap[g0]], c * 256 + kb * 128, grow[g0], &full[st], pol);
              } else {
#pragma unroll
                for (int grp = g0; grp < g0 + 4; ++grp)
                  tma2d_hint(cd + grp * kBox, &p.tm_w[gmap[grp]], c * 256 + kb * 128, grow[grp], &full[st], pol);
              }
            }
          }
#pragma unroll
          for (int hq = 0; hq < 2 && WF == W_FP4; ++hq) {
            const int g0 = 4 * hq;
            if (p.w64 && gmap[g0 + 3] == gmap[g0] && grow[g0 + 3] == grow[g0] + 48) {
              // four groups of one segment: one 64-row code box and one box of
              // their block scales (rows past the matrix are zero-filled)
              tma2d_hint(dst + g0 * kBox, &p.tm_w64[gmap[g0]], c * 128, grow[g0], &full[st], pol);
              tma2d_hint(dst + kCodes + g0 * kScaleBox, &p.tm_s64[gmap[g0]], c * 256, grow[g0] / 16,
                         &full[st], pol);
              continue;
            }
#pragma unroll
            for (int grp = g0; grp < g0 + 4; ++grp) {
              tma2d_hint(dst + grp * kBox, &p.tm_w[gmap[grp]], c * 128, grow[grp], &full[st], pol);
              // block scales of rows 16G .. 16G + 15 and k 256c .. + 255: 256
              // contiguous bytes (groups past the matrix read group 0: their
              // codes are zero-filled)
              const GemmSeg& sg = p.seg[gmap[grp]];
              const int g16 = grow[grp] < sg.rows ? grow[grp] / 16 : 0;
              const char* src = static_cast<const char*>(sg.w) + (size_t)sg.rows * (p.K / 2) +
                                ((size_t)g16 * (p.K / 16) + 16 * c) * 16;
              bulk_hint(dst + kCodes + grp * kScaleBox, src, kScaleBox, &full[st], pol);
            }
          }
          if (!waited) {  // activations may come from the previous kernel
            pdl_wait();
            waited = true;
          }
          if (p.x4) {  // the stage's activations in one copy (same layout)
            tma4d(dst + kCodes + kScales, &p.tm_x4, 0, mb * 16, 0, 4 * c, &full[st]);
          } else {
#pragma unroll
            for (int xb = 0; xb < 4; ++xb) {  // per 64 k: hi rows then lo rows (one 32-row operand)
              tma2d(dst + kCodes + kScales + 2 * xb * kBox, &p.tm_xh, c * 256 + xb * 64, mb * 16, &full[st]);
              tma2d(dst + kCodes + kScales + (2 * xb + 1) * kBox, &p.tm_xl, c * 256 + xb * 64, mb * 16,
                    &full[st]);
            }
          }
        }
      }
      if (p.pf_count > 0) prefetch_share(p, b, G);
      // no copy may still be landing when the CTA exits
      for (long long j = it > kS ? it - kS : 0; j < it; ++j)
        if (!bar_wait(&full[j % kS], (uint32_t)((j / kS) & 1))) {
          atomicOr(p.status, 0x4u);
          break;
        }
    }
  } else if (warp >= kIssuer) {
    // ---------------------------------------------------------------- MMA issuers
    const int iss = warp - kIssuer;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, 32);
      long long it = 0;
      int seg = 0;
      for (long long u = ub0; u < ub1 && !s_abort; ++seg) {
        const int item = (int)(u / p.cpt);
        const int c0 = (int)(u - (long long)item * p.cpt);
        const int c1 = (int)min((long long)p.cpt, c0 + (ub1 - u));
        u += c1 - c0;
        const int db = seg % kDB;
        if (!bar_wait(&acce[db], (uint32_t)((seg / kDB) & 1) ^ 1)) {
          atomicOr(p.status, 0x4u);
          s_abort = 1;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + kDCol + (iss * kDB + db) * 32;
        bool ok = true;
        for (int c = c0; c < c1; ++c, ++it) {
          const int st = (int)(it % kS), ab = (int)(it % kAB);
          if (!bar_wait(&afull[ab], (uint32_t)((it / kAB) & 1)) ||
              !bar_wait(&full[st], (uint32_t)((it / kS) & 1))) {
            atomicOr(p.status, 0x4u);
            s_abort = 1;
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint64_t dx = desc_sw128(su32(sm + st * kStage + kCodes + kScales));
          const uint32_t a = tmem + ab * 128;
#pragma unroll
          for (int s = 16 / kIssuers * iss; s < 16 / kIssuers * (iss + 1); ++s) {
            // B: k16 step s = 32-row box pair s / 4, +32 bytes per step inside its
            // swizzled rows (8-row groups 1024 bytes apart: hi rows 0..15, lo 16..31);
            // the descriptor's address field counts 16-byte units
            const uint32_t boff = (s >> 2) * 2 * kBox + (s & 3) * 32;
            mma_ts(d, a + 8 * s, dx + (boff >> 4), idesc, (c != c0 || s != 16 / kIssuers * iss) ? 1u : 0u);
          }
          commit(&empty[st]);
          commit(&aempty[ab]);
        }
        if (!ok) break;
        commit(&accf[db]);
      }
    }
  } else {
    // ---------------------------------------------------------------- decoders + epilogue
    pdl_wait();   // the epilogues read the previous kernels' outputs
    // warps 8..15 decode (lane quarter q, k half kh of each unit); warps 0..7 run
    // the segment epilogues meanwhile (the next segment's units keep decoding)
    const int q = warp & 3;
    const bool epi = warp < kEpilogue;
    const int h = warp >> 2;    // epilogue warps: column half of the accumulator
    const int kh = (warp >> 2) & 1;
    const int r = 32 * q + lane, grp = r >> 4, rr = r & 15;
    const int pos = 2 * (rr & 7) + (rr >> 3);   // the row's byte in a block of 16 scales
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    long long it = 0;
    int seg = 0;
    for (long long u = ub0; u < ub1; ++seg) {
      const int item = (int)(u / p.cpt);
      const int c0 = (int)(u - (long long)item * p.cpt);
      const int c1 = (int)min((long long)p.cpt, c0 + (ub1 - u));
      u += c1 - c0;
      const int tile = item / p.n_mb, mb = item - tile * p.n_mb;
      for (int c = c0; c < c1 && !epi; ++c, ++it) {
        const int st = (int)(it % kS), ab = (int)(it % kAB);
        if (!s_abort && (!bar_wait(&full[st], (uint32_t)((it / kS) & 1)) ||
                         !bar_wait(&aempty[ab], (uint32_t)((it / kAB) & 1) ^ 1))) {
          if (lane == 0) atomicOr(p.status, 0x4u);
          s_abort = 1;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint8_t* cbox = sm + st * kStage + grp * kBox;
        const uint8_t* sbox = sm + st * kStage + kCodes + grp * kScaleBox + pos;
#pragma unroll
        for (int hf = 0; hf < 2 && WF == W_FP8; ++hf) {
          // this lane's row, 64 k of k half kq / 2: four 16-byte chunks of E4M3
          // codes in natural order, each pair widened to fp16 (exact)
          const int kq = 2 * kh + hf;
          const uint8_t* cb = cbox + (kq >> 1) * (8 * kBox);
          uint4 w4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) w4[i] = *reinterpret_cast<const uint4*>(cb + swz(rr, 4 * (kq & 1) + i));
          uint32_t v[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t ws[4] = {w4[i].x, w4[i].y, w4[i].z, w4[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[8 * i + 2 * e] = e4m3x2_to_f16x2((uint16_t)(ws[e] & 0xffffu));
              v[8 * i + 2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(ws[e] >> 16));
            }
          }
          tmem_st32(tmem + lane_base + ab * 128 + 32 * kq, v);
        }
#pragma unroll
        for (int hf = 0; hf < 2 && WF == W_FP4; ++hf) {
          // this lane's row, k16 steps 4kq .. 4kq + 3: code groups 2kq, 2kq + 1
          // (all loads first)
          const int kq = 2 * kh + hf;
          uint4 w4[2];
          uint32_t sc[4];
#pragma unroll
          for (int g2 = 0; g2 < 2; ++g2) w4[g2] = *reinterpret_cast<const uint4*>(cbox + swz(rr, 2 * kq + g2));
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[e] = sbox[(4 * kq + e) * 16];
          uint32_t v[32];
#pragma unroll
          for (int g2 = 0; g2 < 2; ++g2) {
            const uint32_t s0 = e4m3_pair(sc[2 * g2]), s1 = e4m3_pair(sc[2 * g2 + 1]);
            const uint32_t ws[4] = {w4[g2].x, w4[g2].y, w4[g2].z, w4[g2].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint32_t o[4];
              e2m1x8(ws[t], o);
              // byte 4t + j holds the pair t + 4j of the group (k16 step 2cg + j / 2)
#pragma unroll
              for (int j = 0; j < 4; ++j) v[16 * g2 + t + 4 * j] = hmul2u(o[j], j < 2 ? s0 : s1);
            }
          }
          tmem_st32(tmem + lane_base + ab * 128 + 32 * kq, v);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) bar_arrive(&afull[ab]);
      }
      if (!epi) continue;
      // the segment's accumulators -> acc_s[m][row] = sum over the issuers of
      // D[row][m] + D[row][16 + m] (the hi and lo products): warp (q, h) takes
      // m = 8h .. 8h + 7
      const int db = seg % kDB;
      if (!s_abort && !bar_wait(&accf[db], (uint32_t)((seg / kDB) & 1))) {
        if (lane == 0) atomicOr(p.status, 0x4u);
        s_abort = 1;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      {
        float sum[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sum[e] = 0.f;
#pragma unroll
        for (int i = 0; i < kIssuers; ++i)
#pragma unroll
          for (int hl = 0; hl < 2; ++hl) {
            uint32_t v[8];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                : "r"(tmem + lane_base + kDCol + (i * kDB + db) * 32 + 16 * hl + 8 * h));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int e = 0; e < 8; ++e) sum[e] += __uint_as_float(v[e]);
          }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc_s[(8 * h + e) * kTileRows + r] = sum[e];
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) bar_arrive(&acce[db]);
      if (tid < kTileRows) {
        const float* sc = nullptr;
        const uint8_t* rw = map_row(p, tile, tid, 1, &sc);
        scale_s[tid] = rw ? (sc ? *sc : 1.f) : 0.f;
      }
      if (p.row_scale) compute_inv_rms(p, inv_rms, mb * 16);
      csync();
      if (segment_fixup(p, acc_s, item, c0, c1, U, G, b, &s_flag))
        run_epilogue(p, acc_s, scale_s, inv_rms, mb, tile, &s_flag);
      csync();  // acc_s, scale_s and inv_rms are free for the next segment
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0) stamp_finish(p.stamp);
  if (warp == kIssuer) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols)
                 : "memory");
  }
}

size_t gemm_fp4_smem_bytes() {
  return fp4::Lay<W_FP4>::kSmem > fp4::Lay<W_FP8>::kSmem ? fp4::Lay<W_FP4>::kSmem : fp4::Lay<W_FP8>::kSmem;
}

cudaError_t configure_gemm_fp4() {
  cudaError_t e = cudaFuncSetAttribute(gemm_fp4_kernel<W_FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       fp4::Lay<W_FP4>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_fp4_kernel<W_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             fp4::Lay<W_FP8>::kSmem);
  return e;
}

// p: the schedule of the 16-row kernels (n_tiles, n_mb, cpt = K / 256); the grid
// is one CTA per SM (fewer when there are fewer units).
cudaError_t launch_gemm_fp4(int wt, const GemmParams& p, cudaStream_t st) {
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (n_sm <= 0) n_sm = 1;
  }
  if (!p.has_lo || p.K % 256 != 0) return cudaErrorInvalidValue;
  const long long units = (long long)p.n_tiles * p.n_mb * p.cpt;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units < n_sm ? units : n_sm));
  cfg.blockDim = dim3(fp4::kThreads);
  cfg.dynamicSmemBytes = wt == W_FP8 ? fp4::Lay<W_FP8>::kSmem : fp4::Lay<W_FP4>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (wt == W_FP8) return cudaLaunchKernelEx(&cfg, gemm_fp4_kernel<W_FP8>, p);
  if (wt != W_FP4) return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, gemm_fp4_kernel<W_FP4>, p);
}

}  // namespace dflash
