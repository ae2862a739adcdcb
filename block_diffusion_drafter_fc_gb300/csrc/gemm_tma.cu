// Projection kernel of the block step fed by the Tensor Memory Accelerator.
//
// Same contract as gemm_rows_kernel (y[m][n] = sum_k x[m][k] W[n][k] for 16-row
// activation blocks, stream-K split, fused epilogues) for activations that
// their producer already stored as bf16 hi + lo pairs.  Warps 8 and 9 are
// producers: one lane of each walks this CTA's stream-K units and, per k chunk
// (128 bytes of every weight row), issues cp.async.bulk.tensor loads - warp 8
// of the 128 weight rows, warp 9 of the 16 activation rows (hi and lo) - into a
// ring of shared-memory stages, both completing on the stage's "full" mbarrier.
// The weight rows go as two 64-row
// boxes where four 16-row groups of the tile are consecutive rows of one
// segment (bf16 and E4M3), else as eight 16-row boxes (fp32 weights, segment
// boundaries inside the tile), each from its segment's own tensor map.  Warps 0..7 are consumers: each owns 16 weight rows,
// reads its A fragments and the shared B fragments with ldmatrix from the
// 128-byte-swizzled tiles, runs mma.sync m16n8k16 (fp32 accumulation), and
// releases the stage on its "empty" mbarrier.  The first stages' weight loads
// are issued before griddepcontrol.wait (only the activation warp waits), so
// they overlap the previous kernel.
// Every mbarrier wait gives up after ~2 s, sets the device status bit
// DFLASH_DEV_TIMEOUT and lets the CTA run to completion without further waits;
// before exiting, the producer waits (with the same bound) for its last copies.
#include "gemm_common.cuh"

namespace dflash {

template <int WT>
struct TT;
template <>
struct TT<W_BF16> {  // 64 k per chunk: one 128-byte weight box, one activation box
  static constexpr int CK = 64, WBOX_K = 64, WBOXES = 1, XBOXES = 1, S = 4, STEPS = 4, PEN = 6;
};
template <>
struct TT<W_F32> {   // 64 k per chunk: two 128-byte weight boxes of 32 fp32
  static constexpr int CK = 64, WBOX_K = 32, WBOXES = 2, XBOXES = 1, S = 2, STEPS = 4, PEN = 2;
};
template <>
struct TT<W_FP8> {   // 128 k per chunk: one 128-byte E4M3 box, two activation boxes
  static constexpr int CK = 128, WBOX_K = 128, WBOXES = 1, XBOXES = 2, S = 4, STEPS = 8, PEN = 4;
};

constexpr int kBox = 16 * 128;  // one 16-row x 128-byte box
constexpr long long kWaitCycles = 4000000000LL;

template <int WT>
struct Layout {
  static constexpr int W_BYTES = 8 * kBox * TT<WT>::WBOXES;   // the 8 row groups' weight boxes
  static constexpr int X_BYTES = kBox * TT<WT>::XBOXES;  // one of hi / lo
  static constexpr int STAGE = W_BYTES + 2 * X_BYTES;
  static constexpr int ACC = TT<WT>::S * STAGE;
  static constexpr int INV = ACC + 16 * kTileRows * 4;
  static constexpr int SCALE = INV + 16 * 4;
  static constexpr int BARS = SCALE + kTileRows * 4;
  static constexpr int TOTAL = BARS + 2 * TT<WT>::S * 8 + 1024;  // + alignment slack
};

size_t gemm_tma_smem_bytes(int wt) {
  switch (wt) {
    case W_F32: return Layout<W_F32>::TOTAL;
    case W_BF16: return Layout<W_BF16>::TOTAL;
    case W_FP8: return Layout<W_FP8>::TOTAL;
  }
  return 0;
}

// ------------------------------------------------------------------ primitives

DF_DEVICE uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

DF_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count) : "memory");
}
DF_DEVICE void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes)
               : "memory");
}
DF_DEVICE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
DF_DEVICE bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(su32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for completion of the phase with this parity; false after ~2 s.
DF_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}

DF_DEVICE void tma_load(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}

// The same load with an L2 eviction-priority hint (weights: read once per step,
// so they should not push the activations, partials and ring out of L2).
DF_DEVICE void tma_load_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(su32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(su32(bar)), "l"(policy)
      : "memory");
}
DF_DEVICE uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

DF_DEVICE void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(su32(p)));
}

// byte offset of (row, 16-byte chunk) inside a 128-byte-swizzled box
DF_DEVICE int swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

// ------------------------------------------------------------------ consumer math

template <int WT>
struct Consume;

// B fragments (two n8 tiles) of k16 step `kc2` (16-byte chunk pair index) from
// one activation box
DF_DEVICE void x_frags(uint32_t (&b)[4], const uint8_t* box, int kchunk0, int lane) {
  const int lmat = lane >> 3, lrow = lane & 7;
  const int row = (lmat >> 1) * 8 + lrow, chunk = kchunk0 + (lmat & 1);
  ldsm_x4(b, box + swz(row, chunk));
}

template <>
struct Consume<W_BF16> {
  static DF_DEVICE void run(const uint8_t* w, const uint8_t* xh, const uint8_t* xl, bool has_lo,
                            int lane, float (&acc)[2][4]) {
    const int lmat = lane >> 3, lrow = lane & 7;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a[4], b[4];
      const int arow = (lmat & 1) * 8 + lrow;
      ldsm_x4(a, w + swz(arow, 2 * s + (lmat >> 1)));
      x_frags(b, xh, 2 * s, lane);
      mma_bf16_16816(acc[0], a, b[0], b[1]);
      mma_bf16_16816(acc[1], a, b[2], b[3]);
      if (has_lo) {
        x_frags(b, xl, 2 * s, lane);
        mma_bf16_16816(acc[0], a, b[0], b[1]);
        mma_bf16_16816(acc[1], a, b[2], b[3]);
      }
    }
  }
};

template <>
struct Consume<W_FP8> {
  static DF_DEVICE void run(const uint8_t* w, const uint8_t* xh, const uint8_t* xl, bool has_lo,
                            int lane, float (&acc)[2][4]) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      // E4M3 pairs (k = 16s + 2t and + 8) of rows g and g + 8, widened to fp16
      // (exact, one conversion each); the activations are an fp16 hi/lo pair
      const uint16_t q0 = *reinterpret_cast<const uint16_t*>(w + swz(g, s) + 2 * t);
      const uint16_t q1 = *reinterpret_cast<const uint16_t*>(w + swz(g + 8, s) + 2 * t);
      const uint16_t q2 = *reinterpret_cast<const uint16_t*>(w + swz(g, s) + 2 * t + 8);
      const uint16_t q3 = *reinterpret_cast<const uint16_t*>(w + swz(g + 8, s) + 2 * t + 8);
      const uint32_t a[4] = {e4m3x2_to_f16x2(q0), e4m3x2_to_f16x2(q1), e4m3x2_to_f16x2(q2),
                             e4m3x2_to_f16x2(q3)};
      uint32_t b[4];
      x_frags(b, xh + (s >> 2) * kBox, 2 * (s & 3), lane);
      mma_f16_16816(acc[0], a, b[0], b[1]);
      mma_f16_16816(acc[1], a, b[2], b[3]);
      if (has_lo) {
        x_frags(b, xl + (s >> 2) * kBox, 2 * (s & 3), lane);
        mma_f16_16816(acc[0], a, b[0], b[1]);
        mma_f16_16816(acc[1], a, b[2], b[3]);
      }
    }
  }
};

template <>
struct Consume<W_F32> {
  static DF_DEVICE void run(const uint8_t* w, const uint8_t* xh, const uint8_t* xl, bool has_lo,
                            int lane, float (&acc)[2][4]) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      // fp32 pairs of rows g, g + 8 at k = 16s + 2t (+8): box s/2, byte 64(s&1) + 8t (+32)
      const uint8_t* bx = w + (s >> 1) * kBox;
      const int byte0 = 64 * (s & 1) + 8 * t, byte1 = byte0 + 32;
      const float2 f0 = *reinterpret_cast<const float2*>(bx + swz(g, byte0 >> 4) + (byte0 & 15));
      const float2 f1 = *reinterpret_cast<const float2*>(bx + swz(g + 8, byte0 >> 4) + (byte0 & 15));
      const float2 f2 = *reinterpret_cast<const float2*>(bx + swz(g, byte1 >> 4) + (byte1 & 15));
      const float2 f3 = *reinterpret_cast<const float2*>(bx + swz(g + 8, byte1 >> 4) + (byte1 & 15));
      uint32_t ah[4], al[4];
      split_bf16x2(f0.x, f0.y, ah[0], al[0]);
      split_bf16x2(f1.x, f1.y, ah[1], al[1]);
      split_bf16x2(f2.x, f2.y, ah[2], al[2]);
      split_bf16x2(f3.x, f3.y, ah[3], al[3]);
      uint32_t b[4];
      x_frags(b, xh, 2 * s, lane);
      mma_bf16_16816(acc[0], ah, b[0], b[1]);
      mma_bf16_16816(acc[1], ah, b[2], b[3]);
      mma_bf16_16816(acc[0], al, b[0], b[1]);
      mma_bf16_16816(acc[1], al, b[2], b[3]);
      if (has_lo) {
        x_frags(b, xl, 2 * s, lane);
        mma_bf16_16816(acc[0], ah, b[0], b[1]);
        mma_bf16_16816(acc[1], ah, b[2], b[3]);
      }
    }
  }
};

// ------------------------------------------------------------------ kernel

// Tensor-map index and row coordinate of 16-row group `grp` of `tile`: rows past
// the matrix are addressed out of bounds, which the copy fills with zeros.
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

// Stream-K split over a weighted axis.  A CTA whose range crosses into a new
// item stops its chunk stream for that item's partial publication (stores made
// visible at GPU scope, then the ticket), which costs it about as long as
// streaming PEN chunks.  So every item is PEN + cpt units long on the split
// axis - PEN for the crossing, then its cpt chunks - and the G CTAs share that
// axis equally: the CTAs that cross an item boundary get fewer chunks.
// Chunk unit of split position v (a position inside an item's crossing part
// maps to the item's first chunk).
DF_DEVICE long long vsplit_unit(long long v, int cpt, int pen) {
  const long long i = v / (cpt + pen), r = v - i * (cpt + pen);
  return i * cpt + (r > pen ? r - pen : 0);
}
// The CTA whose range holds chunk unit u.
DF_DEVICE int vsplit_owner(long long u, int cpt, int pen, long long V, int G) {
  const long long i = u / cpt, v = i * (cpt + pen) + pen + (u - i * cpt);
  return (int)(((v + 1) * G - 1) / V);
}

// segment_fixup for the weighted split: after a segment [c0, c1) of `item` has
// been accumulated into acc_s, publish it if the tile is shared and, for the
// last contributor (acquire-release ticket), sum all partials in CTA order.
// Returns true when this CTA must run the tile's epilogue.
template <int PEN>
DF_DEVICE bool vsplit_fixup(const GemmParams& p, float* acc_s, int item, int c0, int c1,
                            long long V, int G, int b, int* s_flag) {
  constexpr int kVec = 16 * kTileRows / 4;  // float4 per partial tile
  constexpr int kPer = kVec / kGemmThreads;  // float4 per thread
  constexpr int kBatch = 4;
  const int tid = threadIdx.x;
  if (c0 == 0 && c1 == p.cpt) return true;
  const long long iu0 = (long long)item * p.cpt;
  const int first = vsplit_owner(iu0, p.cpt, PEN, V, G);
  const int last = vsplit_owner(iu0 + p.cpt - 1, p.cpt, PEN, V, G);
  float4* acc4 = reinterpret_cast<float4*>(acc_s);
  auto part_of = [&](int c) {
    const size_t sl = 2 * (size_t)c + (c == first ? 1 : 0);
    return reinterpret_cast<float4*>(p.partial + sl * (16 * kTileRows));
  };
  float4* mine = part_of(b);
#pragma unroll
  for (int k = 0; k < kPer; ++k) __stcg(mine + tid + k * kGemmThreads, acc4[tid + k * kGemmThreads]);
  csync();
  if (tid == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(p.counters + item)
                 : "memory");
    *s_flag = old == last - first;
  }
  csync();
  if (!*s_flag) return false;
  float4 sum[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) sum[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int cb = first; cb <= last; cb += kBatch) {
    float4 v[kBatch][kPer];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (cb + j <= last) v[j][k] = __ldcg(part_of(cb + j) + tid + k * kGemmThreads);
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (cb + j <= last) {
          sum[k].x += v[j][k].x;
          sum[k].y += v[j][k].y;
          sum[k].z += v[j][k].z;
          sum[k].w += v[j][k].w;
        }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc4[tid + k * kGemmThreads] = sum[k];
  if (tid == 0) p.counters[item] = 0;
  csync();
  return true;
}

// This CTA's 1/G share of the prefetch ranges (16-byte aligned pieces of at
// most 32 KB): the next kernel's input moves into L2 while this kernel's last
// weight stages are still streaming.
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

// ------------------------------------------------------------------ chains

DF_DEVICE int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
DF_DEVICE void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DF_DEVICE void red_release_add_gpu(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DF_DEVICE int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// This CTA's range of a phase on the weighted stream-K axis (chunk units).  A
// phase is split over its own p.grid CTAs (no more than it has chunk units, as
// a launch of that projection alone would be); CTAs past them sit it out.
template <int PEN>
DF_DEVICE void phase_range(const GemmParams& p, int b, long long& V, long long& u0, long long& u1) {
  V = (long long)p.n_tiles * p.n_mb * (p.cpt + PEN);
  if (b >= p.grid) {
    u0 = u1 = 0;
    return;
  }
  u0 = vsplit_unit(V * b / p.grid, p.cpt, PEN);
  u1 = vsplit_unit(V * (b + 1) / p.grid, p.cpt, PEN);
}

template <int WT, int NPH>
__global__ void __launch_bounds__(kGemmThreads + 64, 2)
    gemm_tma_kernel(const __grid_constant__ ChainParams<NPH> cp) {
  using T = TT<WT>;
  using Lt = Layout<WT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* acc_s = reinterpret_cast<float*>(sm + Lt::ACC);
  float* inv_rms = reinterpret_cast<float*>(sm + Lt::INV);
  float* scale_s = reinterpret_cast<float*>(sm + Lt::SCALE);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lt::BARS);
  uint64_t* empty = full + T::S;
  __shared__ int s_flag;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_ph = NPH == 1 ? 1 : cp.n_phase;
  if (tid == 0) {
    for (int s = 0; s < T::S; ++s) {
      mbar_init(&full[s], 2);   // one arrival from each producer warp
      mbar_init(&empty[s], 8);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    stamp_begin(cp.ph[0].stamp);
  }
  __syncthreads();
  pdl_trigger();

  const int G = gridDim.x, b = blockIdx.x;

  if (warp >= 8) {
    // ------------------------------------------------------------ producers
    // Two producer warps, one thread each: warp 8 issues the weight boxes,
    // warp 9 the activation boxes (the stream is issue-bound on one thread).
    // Both walk the CTA's chunks of phase 0, 1, ... in the same order (chunk g
    // uses stage g % S, whose "full" barrier takes one arrival from each, with
    // the bytes it expects) and wait for the stage to be free.  Only the
    // activation warp waits for inputs: the previous kernel (phase 0) or the
    // previous phase's items (chains); the weight warp runs up to S chunks ahead.
    if (lane != 0) return;
    const bool wwarp = warp == 8;
    const uint64_t w_policy = policy_evict_first();
    int ph = 0, item = 0, c = 0, tile = 0, mb = 0;
    long long j = 0, n = 0;
    auto begin_phase = [&](int k) {
      const GemmParams& p = cp.ph[k];
      long long V, u0, u1;
      phase_range<T::PEN>(p, b, V, u0, u1);
      ph = k;
      j = 0;
      n = u1 - u0;
      item = (int)(u0 / p.cpt);
      c = (int)(u0 - (long long)item * p.cpt);
      tile = item / p.n_mb;
      mb = item - tile * p.n_mb;
    };
    begin_phase(0);
    while (j >= n && ph + 1 < n_ph) begin_phase(ph + 1);
    int gmap[8], grow[8], g_tile = -1, g_ph = -1;
    long long g = 0;
    bool abort = false;
    int ready_ph = 0;   // a phase whose inputs are all complete (no more checks)
    if (!wwarp) pdl_wait();   // phase 0's activations come from the previous kernel
    for (; j < n; ++g) {
      const GemmParams& p = cp.ph[ph];
      const int st = (int)(g % T::S);
      if (g >= T::S && !abort && !mbar_wait(&empty[st], (uint32_t)(((g / T::S) & 1) ^ 1))) {
        atomicOr(p.status, 0x4u);
        abort = true;   // keep arming and issuing (unchecked) so every stage completes
        s_abort = 1;
      }
      uint8_t* dst = sm + st * Lt::STAGE;
      if (wwarp) {
        if (tile != g_tile || ph != g_ph) {
#pragma unroll
          for (int grp = 0; grp < 8; ++grp) group_coord(p, tile, grp, gmap[grp], grow[grp]);
          g_tile = tile;
          g_ph = ph;
        }
        const int k = c * T::CK;
        mbar_expect_tx(&full[st], Lt::W_BYTES);
        if (T::WBOXES == 1 && p.w64) {
          // four 16-row groups of one segment with consecutive rows are one
          // 64-row box (the same swizzled layout as four stacked 16-row boxes)
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            const int g0 = 4 * hq;
            if (gmap[g0 + 3] == gmap[g0] && grow[g0 + 3] == grow[g0] + 48) {
              tma_load_hint(dst + g0 * kBox, &p.tm_w64[gmap[g0]], k, grow[g0], &full[st], w_policy);
            } else {
#pragma unroll
              for (int grp = g0; grp < g0 + 4; ++grp)
                tma_load_hint(dst + grp * kBox, &p.tm_w[gmap[grp]], k, grow[grp], &full[st], w_policy);
            }
          }
        } else {
#pragma unroll
          for (int grp = 0; grp < 8; ++grp)
#pragma unroll
            for (int wb = 0; wb < T::WBOXES; ++wb)
              tma_load_hint(dst + (grp * T::WBOXES + wb) * kBox, &p.tm_w[gmap[grp]],
                            k + wb * T::WBOX_K, grow[grp], &full[st], w_policy);
        }
      } else {
        if (NPH > 1 && ph > 0 && !abort && ready_ph != ph) {
          // phase ph reads phase ph - 1's output columns [k0, k0 + CK) of this
          // 16-row block: wait for the items that write them (acquire); once
          // every item of the block is done, the rest of the phase needs no check
          const GemmParams& pp = cp.ph[ph - 1];
          const int* cnt = cp.all_done + (size_t)(ph - 1) * cp.mb_stride + mb;
          if (ld_acquire_gpu(cnt) >= pp.n_tiles) {
            if (pp.n_mb == 1) ready_ph = ph;
          } else {
            const int tc = pp.map == MAP_SWIGLU ? kTileRows / 2 : kTileRows;
            const int k0 = c * T::CK;
            const int* flags = cp.item_done + (size_t)(ph - 1) * cp.item_stride;
            for (int t = k0 / tc; t <= (k0 + T::CK - 1) / tc && !abort; ++t) {
              const int* f = flags + t * pp.n_mb + mb;
              const long long t0 = clock64();
              while (!ld_acquire_gpu(f)) {
                __nanosleep(64);
                if (clock64() - t0 > kWaitCycles) {
                  atomicOr(p.status, 0x4u);
                  abort = true;
                  s_abort = 1;
                  break;
                }
              }
            }
          }
          // the tensor copies (async proxy) read what the epilogues' plain stores wrote
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const int k = c * T::CK;
        mbar_expect_tx(&full[st], Lt::X_BYTES * (p.has_lo ? 2 : 1));
#pragma unroll
        for (int xb = 0; xb < T::XBOXES; ++xb) {
          tma_load(dst + Lt::W_BYTES + xb * kBox, &p.tm_xh, k + xb * 64, mb * 16, &full[st]);
          if (p.has_lo)
            tma_load(dst + Lt::W_BYTES + Lt::X_BYTES + xb * kBox, &p.tm_xl, k + xb * 64, mb * 16,
                     &full[st]);
        }
      }
      // next chunk
      ++j;
      if (++c == p.cpt) {
        c = 0;
        ++item;
        if (++mb == p.n_mb) {
          mb = 0;
          ++tile;
        }
      }
      while (j >= n && ph + 1 < n_ph) begin_phase(ph + 1);
    }
    if (wwarp)
      for (int k = 0; k < n_ph; ++k)
        if (cp.ph[k].pf_count > 0) prefetch_share(cp.ph[k], b, G);
    // no copy of this warp may still be landing when the CTA exits
    for (long long q = g > T::S ? g - T::S : 0; q < g; ++q) {
      if (!mbar_wait(&full[q % T::S], (uint32_t)((q / T::S) & 1))) {
        atomicOr(cp.ph[0].status, 0x4u);
        break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  long long it = 0;
  for (int ph = 0; ph < n_ph; ++ph) {
    const GemmParams& p = cp.ph[ph];
    const bool has_lo = p.has_lo != 0;
    long long V, ub0, ub1;
    phase_range<T::PEN>(p, b, V, ub0, ub1);
    for (long long u = ub0; u < ub1;) {
      const int item = (int)(u / p.cpt);
      const int c0 = (int)(u - (long long)item * p.cpt);
      const int c1 = (int)min((long long)p.cpt, c0 + (ub1 - u));
      u += c1 - c0;
      const int tile = item / p.n_mb, mb = item - tile * p.n_mb;
      csync();  // the previous segment is done with acc_s / scale_s / inv_rms
      if (tid < kTileRows) {
        const float* sc = nullptr;
        const uint8_t* r = map_row(p, tile, tid, 1, &sc);
        scale_s[tid] = r ? (sc ? *sc : 1.f) : 0.f;
      }
      // the row statistics of phase 0 come from an earlier kernel
      if (p.row_scale && ph == 0) compute_inv_rms(p, inv_rms, mb * 16);
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      for (int c = c0; c < c1; ++c, ++it) {
        const int st = (int)(it % T::S);
        if (!s_abort) {
          if (mbar_wait(&full[st], (uint32_t)((it / T::S) & 1))) {
            const uint8_t* base = sm + st * Lt::STAGE;
            Consume<WT>::run(base + warp * T::WBOXES * kBox, base + Lt::W_BYTES,
                             base + Lt::W_BYTES + Lt::X_BYTES, has_lo, lane, acc);
          } else {
            if (lane == 0) atomicOr(p.status, 0x4u);
            s_abort = 1;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      const int g = lane >> 2, t = lane & 3;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int cc = 8 * j + 2 * t, r = warp * 16 + g;
        acc_s[cc * kTileRows + r] = acc[j][0];
        acc_s[(cc + 1) * kTileRows + r] = acc[j][1];
        acc_s[cc * kTileRows + r + 8] = acc[j][2];
        acc_s[(cc + 1) * kTileRows + r + 8] = acc[j][3];
      }
      csync();
      if (!vsplit_fixup<T::PEN>(p, acc_s, item, c0, c1, V, p.grid, b, &s_flag)) continue;
      if (p.row_scale && ph > 0) {
        // the 1/rms of the block's rows needs every item of the previous phase
        // in this 16-row block (their sums of squares): wait (bounded), then read
        if (tid == 0) {
          const int* cnt = cp.all_done + (size_t)(ph - 1) * cp.mb_stride + mb;
          const long long t0 = clock64();
          while (ld_acquire_gpu(cnt) < cp.ph[ph - 1].n_tiles && !s_abort) {
            __nanosleep(64);
            if (clock64() - t0 > kWaitCycles) {
              atomicOr(p.status, 0x4u);
              s_abort = 1;
            }
          }
        }
        csync();
        compute_inv_rms(p, inv_rms, mb * 16);
        csync();
      }
      run_epilogue(p, acc_s, scale_s, inv_rms, mb, tile, &s_flag);
      if (NPH > 1 && ph + 1 < n_ph) {
        csync();  // every thread's epilogue stores precede the release
        if (tid == 0) {
          st_release_gpu(cp.item_done + (size_t)ph * cp.item_stride + item, 1);
          red_release_add_gpu(cp.all_done + (size_t)ph * cp.mb_stride + mb, 1);
        }
      }
    }
  }
  csync();
  if (tid == 0) {
    stamp_finish(cp.ph[0].stamp);
    if (NPH > 1) s_flag = atom_add_acq_rel_gpu(cp.chain_done, 1) == G - 1;
  }
  if (NPH > 1) {
    // the last CTA past the chain clears the flags and counters for the next
    // launch (every CTA's producer read its last flag before its last chunk)
    csync();
    if (s_flag) {
      const int n_items = (n_ph - 1) * cp.item_stride, n_mbs = (n_ph - 1) * cp.mb_stride;
      for (int i = tid; i < n_items; i += kGemmThreads) cp.item_done[i] = 0;
      for (int i = tid; i < n_mbs; i += kGemmThreads) cp.all_done[i] = 0;
      if (tid == 0) *cp.chain_done = 0;
    }
  }
}

template <int WT, int NPH>
static cudaError_t set_smem() {
  return cudaFuncSetAttribute(gemm_tma_kernel<WT, NPH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)gemm_tma_smem_bytes(WT));
}

cudaError_t configure_gemm_tma() {
  cudaError_t e = set_smem<W_F32, 1>();
  if (e == cudaSuccess) e = set_smem<W_BF16, 1>();
  if (e == cudaSuccess) e = set_smem<W_FP8, 1>();
  if (e == cudaSuccess) e = set_smem<W_F32, kChainMax>();
  if (e == cudaSuccess) e = set_smem<W_BF16, kChainMax>();
  if (e == cudaSuccess) e = set_smem<W_FP8, kChainMax>();
  return e;
}

template <int WT, int NPH>
static cudaError_t launch_tma_t(const ChainParams<NPH>& cp, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads + 64);
  cfg.dynamicSmemBytes = gemm_tma_smem_bytes(WT);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tma_kernel<WT, NPH>, cp);
}

cudaError_t launch_gemm_tma(int wt, const GemmParams& p, cudaStream_t st) {
  ChainParams<1> cp;
  cp.ph[0] = p;
  cp.n_phase = 1;
  cp.item_done = cp.all_done = cp.chain_done = nullptr;
  cp.item_stride = cp.mb_stride = 0;
  switch (wt) {
    case W_F32: return launch_tma_t<W_F32, 1>(cp, p.grid, st);
    case W_BF16: return launch_tma_t<W_BF16, 1>(cp, p.grid, st);
    case W_FP8: return launch_tma_t<W_FP8, 1>(cp, p.grid, st);
  }
  return cudaErrorInvalidValue;
}

template <int WT>
static int chain_capacity_t() {
  int per_sm = 0, dev = 0, n_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_tma_kernel<WT, kChainMax>, kGemmThreads + 64,
                                                    gemm_tma_smem_bytes(WT)) != cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return per_sm * n_sm;
}

int gemm_chain_capacity(int wt) {
  switch (wt) {
    case W_F32: return chain_capacity_t<W_F32>();
    case W_BF16: return chain_capacity_t<W_BF16>();
    case W_FP8: return chain_capacity_t<W_FP8>();
  }
  return 0;
}

// the chain's grid: the largest of its phases' grids
cudaError_t launch_gemm_chain(int wt, const ChainParams<kChainMax>& cp, cudaStream_t st) {
  int grid = 0;
  for (int k = 0; k < cp.n_phase; ++k) grid = cp.ph[k].grid > grid ? cp.ph[k].grid : grid;
  switch (wt) {
    case W_F32: return launch_tma_t<W_F32, kChainMax>(cp, grid, st);
    case W_BF16: return launch_tma_t<W_BF16, kChainMax>(cp, grid, st);
    case W_FP8: return launch_tma_t<W_FP8, kChainMax>(cp, grid, st);
  }
  return cudaErrorInvalidValue;
}

// (FP4 weights: the 256-k units of the FP4 kernel)
int tma_chunk_k(int wt) { return wt == W_FP4 ? 256 : wt == W_FP8 ? 128 : 64; }

}  // namespace dflash
