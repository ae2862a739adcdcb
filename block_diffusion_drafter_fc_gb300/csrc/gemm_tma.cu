// Projection kernel of the block step fed by the Tensor Memory Accelerator.
//
// Same contract as gemm_rows_kernel (y[m][n] = sum_k x[m][k] W[n][k] for 16-row
// activation blocks, stream-K split, fused epilogues) for activations that
// their producer already stored as bf16 hi + lo pairs.  Warp 8 is a producer:
// one lane walks this CTA's stream-K units and, per k chunk (128 bytes of every
// weight row), issues cp.async.bulk.tensor loads of the 128 weight rows and of
// the 16 activation rows (hi and lo) into a ring of shared-memory stages,
// completing on the stage's "full" mbarrier.  The weight rows go as two 64-row
// boxes where four 16-row groups of the tile are consecutive rows of one
// segment (bf16 and E4M3), else as eight 16-row boxes (fp32 weights, segment
// boundaries inside the tile), each from its segment's own tensor map.  Warps 0..7 are consumers: each owns 16 weight rows,
// reads its A fragments and the shared B fragments with ldmatrix from the
// 128-byte-swizzled tiles, runs mma.sync m16n8k16 (fp32 accumulation), and
// releases the stage on its "empty" mbarrier.  The first stages' weight loads
// are issued before griddepcontrol.wait, so they overlap the previous kernel.
// Every mbarrier wait gives up after ~2 s, sets the device status bit
// DFLASH_DEV_TIMEOUT and lets the CTA run to completion without further waits;
// before exiting, the producer waits (with the same bound) for its last copies.
#include "gemm_common.cuh"

namespace dflash {

template <int WT>
struct TT;
template <>
struct TT<W_BF16> {  // 64 k per chunk: one 128-byte weight box, one activation box
  static constexpr int CK = 64, WBOX_K = 64, WBOXES = 1, XBOXES = 1, S = 4, STEPS = 4, PEN = 4;
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
      // E4M3 pairs (k = 16s + 2t and + 8) of rows g and g + 8, widened to bf16
      const uint16_t q0 = *reinterpret_cast<const uint16_t*>(w + swz(g, s) + 2 * t);
      const uint16_t q1 = *reinterpret_cast<const uint16_t*>(w + swz(g + 8, s) + 2 * t);
      const uint16_t q2 = *reinterpret_cast<const uint16_t*>(w + swz(g, s) + 2 * t + 8);
      const uint16_t q3 = *reinterpret_cast<const uint16_t*>(w + swz(g + 8, s) + 2 * t + 8);
      const uint32_t a[4] = {e4m3x2_to_bf16x2(q0), e4m3x2_to_bf16x2(q1), e4m3x2_to_bf16x2(q2),
                             e4m3x2_to_bf16x2(q3)};
      uint32_t b[4];
      x_frags(b, xh + (s >> 2) * kBox, 2 * (s & 3), lane);
      mma_bf16_16816(acc[0], a, b[0], b[1]);
      mma_bf16_16816(acc[1], a, b[2], b[3]);
      if (has_lo) {
        x_frags(b, xl + (s >> 2) * kBox, 2 * (s & 3), lane);
        mma_bf16_16816(acc[0], a, b[0], b[1]);
        mma_bf16_16816(acc[1], a, b[2], b[3]);
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

template <int WT>
__global__ void __launch_bounds__(kGemmThreads + 32, 2) gemm_tma_kernel(const __grid_constant__ GemmParams p) {
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
  if (tid == 0) {
    for (int s = 0; s < T::S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    stamp_begin(p.stamp);
  }
  __syncthreads();
  pdl_trigger();

  const int G = gridDim.x, b = blockIdx.x;
  const long long V = (long long)p.n_tiles * p.n_mb * (p.cpt + T::PEN);
  const long long ub0 = vsplit_unit(V * b / G, p.cpt, T::PEN),
                  ub1 = vsplit_unit(V * (b + 1) / G, p.cpt, T::PEN);
  const bool has_lo = p.has_lo != 0;
  const uint32_t stage_bytes = Lt::W_BYTES + Lt::X_BYTES * (has_lo ? 2 : 1);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // One thread issues every copy, so its per-chunk work stays a handful of
    // instructions: two cursors walk the CTA's chunks (the weights' one ahead
    // of the activations' one during the prologue) with one division per item.
    if (lane != 0) return;
    const uint64_t w_policy = policy_evict_first();
    const long long n = ub1 - ub0;   // k chunks of this CTA
    struct Cursor {
      int item, c, tile, mb;
    };
    auto start = [&](Cursor& q) {
      q.item = (int)(ub0 / p.cpt);
      q.c = (int)(ub0 - (long long)q.item * p.cpt);
      q.tile = q.item / p.n_mb;
      q.mb = q.item - q.tile * p.n_mb;
    };
    auto advance = [&](Cursor& q) {
      if (++q.c == p.cpt) {
        q.c = 0;
        ++q.item;
        if (++q.mb == p.n_mb) {
          q.mb = 0;
          ++q.tile;
        }
      }
    };
    Cursor cw, cx;
    start(cw);
    start(cx);
    int gmap[8], grow[8], g_tile = -1;
    // the weight boxes of the chunk at cursor cw into stage st (arming the
    // stage's barrier for the whole stage)
    auto issue_w = [&](int st) {
      if (cw.tile != g_tile) {
#pragma unroll
        for (int grp = 0; grp < 8; ++grp) group_coord(p, cw.tile, grp, gmap[grp], grow[grp]);
        g_tile = cw.tile;
      }
      uint8_t* dst = sm + st * Lt::STAGE;
      const int k = cw.c * T::CK;
      mbar_expect_tx(&full[st], stage_bytes);
      if (T::WBOXES == 1 && p.w64) {
        // four 16-row groups of one segment with consecutive rows are one
        // 64-row box (the same swizzled layout as four stacked 16-row boxes):
        // fewer, larger copies
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
      advance(cw);
    };
    // the activation boxes (hi, lo) of the chunk at cursor cx into stage st
    auto issue_x = [&](int st) {
      uint8_t* dst = sm + st * Lt::STAGE;
      const int k = cx.c * T::CK;
#pragma unroll
      for (int xb = 0; xb < T::XBOXES; ++xb) {
        tma_load(dst + Lt::W_BYTES + xb * kBox, &p.tm_xh, k + xb * 64, cx.mb * 16, &full[st]);
        if (has_lo)
          tma_load(dst + Lt::W_BYTES + Lt::X_BYTES + xb * kBox, &p.tm_xl, k + xb * 64, cx.mb * 16,
                   &full[st]);
      }
      advance(cx);
    };
    // Weights do not depend on the previous kernel: every stage's weight boxes
    // go out before the dependency wait, so the stream is already in flight
    // when the activations become readable; then those stages' activations.
    const int pre = n < T::S ? (int)n : T::S;
    for (int j = 0; j < pre; ++j) issue_w(j);
    pdl_wait();
    for (int j = 0; j < pre; ++j) issue_x(j);
    long long it = pre;
    int st = pre % T::S;
    uint32_t ph = pre / T::S;   // 0 or 1: the parity of chunk `it`'s stage round
    for (; it < n && !s_abort; ++it) {
      if (!mbar_wait(&empty[st], (ph & 1) ^ 1)) {
        atomicOr(p.status, 0x4u);
        s_abort = 1;
        break;
      }
      issue_w(st);
      issue_x(st);
      if (++st == T::S) {
        st = 0;
        ++ph;
      }
    }
    if (p.pf_count > 0) prefetch_share(p, b, G);
    // no copy may still be landing when the CTA exits: wait for the last stages
    for (long long j = it > T::S ? it - T::S : 0; j < it; ++j) {
      if (!mbar_wait(&full[j % T::S], (uint32_t)((j / T::S) & 1))) {
        atomicOr(p.status, 0x4u);
        break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  {
    long long it = 0;
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
      if (p.row_scale) compute_inv_rms(p, inv_rms, mb * 16);
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
      if (!vsplit_fixup<T::PEN>(p, acc_s, item, c0, c1, V, G, b, &s_flag)) continue;
      run_epilogue(p, acc_s, scale_s, inv_rms, mb, tile, &s_flag);
    }
  }
  if (p.stamp) {
    csync();
    if (tid == 0) stamp_finish(p.stamp);
  }
}

cudaError_t configure_gemm_tma() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tma_kernel<W_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gemm_tma_smem_bytes(W_F32));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tma_kernel<W_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gemm_tma_smem_bytes(W_BF16));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tma_kernel<W_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gemm_tma_smem_bytes(W_FP8));
  return e;
}

template <int WT>
static cudaError_t launch_tma_t(const GemmParams& p, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kGemmThreads + 32);
  cfg.dynamicSmemBytes = gemm_tma_smem_bytes(WT);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kDependentLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tma_kernel<WT>, p);
}

cudaError_t launch_gemm_tma(int wt, const GemmParams& p, cudaStream_t st) {
  switch (wt) {
    case W_F32: return launch_tma_t<W_F32>(p, st);
    case W_BF16: return launch_tma_t<W_BF16>(p, st);
    case W_FP8: return launch_tma_t<W_FP8>(p, st);
  }
  return cudaErrorInvalidValue;
}

// (FP4 weights: the 256-k units of the FP4 kernel)
int tma_chunk_k(int wt) { return wt == W_FP4 ? 256 : wt == W_FP8 ? 128 : 64; }

}  // namespace dflash
