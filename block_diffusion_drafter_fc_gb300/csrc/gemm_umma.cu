// Dense projection kernel on the 5th-generation tensor cores (tcgen05), for
// steps with at least 128 activation rows (the cross-sequence batch of
// dflash_head.rs, struct DflashBatch: 16 rows per sequence).
//
// Persistent: one CTA per SM walks output tiles D[128 activation rows][WR
// weight rows] (WR = 128 or 256; tile t = CTA, CTA + grid, ...; consecutive
// tiles share a weight tile across the activation row blocks, so weights come
// from HBM once), each over the whole k range, with the accumulator
// double-buffered in tensor memory so that a tile's epilogue overlaps the next
// tile's MMAs:
//   warp 12 (one lane)  TMA producer: per 64-wide k chunk, the activation hi and
//                       lo boxes [128 rows x 128 B] and the weight boxes into a
//                       3- or 4-stage shared-memory ring (128-byte swizzle, the
//                       UMMA K-major canonical layout), across tile boundaries,
//                       and an L2 prefetch of the weights kPf chunks ahead;
//   warps 8..11         E4M3 weights only: widen the raw [WR x 64] byte tile to
//                       the bf16 swizzled tile the MMA reads (exact), then fence
//                       the generic-proxy writes for the async proxy;
//   warp 13 (one lane)  allocates 2 x WR TMEM columns and issues, per k16 step,
//                       tcgen05.mma kind::f16 (bf16 x bf16, fp32 accumulate) for
//                       the activation hi part and again for the lo part (the
//                       fp32 activations are split into bf16 hi + lo) into the
//                       tile's accumulator buffer; commits each stage back to
//                       the producer and each finished tile to the epilogue;
//   warps 0..7          the fused epilogues of the 16-row kernels (RMS row
//                       scale, per-head q/k norm + rope, residual + next input,
//                       SwiGLU, logits + argmax): one thread per activation row
//                       straight from tensor memory (tcgen05.ld), or per 16-row
//                       block through shared memory for the ring injection;
//                       then hand the buffer back to the MMA.
// Every mbarrier wait gives up after ~2 s with DFLASH_DEV_TIMEOUT; tensor memory
// is always released before exit.
#include "gemm_common.cuh"

namespace dflash {

namespace umma {

constexpr int kTile = 128 * 128;       // bytes of one [128 rows x 128 B] swizzled tile
constexpr long long kWait = 4000000000LL;
constexpr int kThreads = 448;          // warps 0-7 epilogue, 8-11 E4M3 widening, 12 TMA, 13 MMA
constexpr int kWiden = 4;              // widening warps
constexpr int kBRow = kTileRows + 4;   // padded row (floats) of a read-out block
constexpr int kPf = 6;                 // weight chunks prefetched into L2 ahead of the box loads

// Shared-memory layout for output tiles of 128 activation rows x WR weight rows
// (WR = 128, or 256 = two 128-row n-tiles sharing every activation chunk).
template <int WR>
struct L {
  // pipeline stages: as many as shared memory holds next to the epilogue scratch
  static constexpr int kS = WR == 128 ? 4 : 3;
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

DF_DEVICE void tma_prefetch2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
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

// 16 consecutive fp32 accumulator columns of the warp's 32 tensor-memory lanes
// (lane i: activation row i of the warp's quadrant)
DF_DEVICE void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  __syncwarp();   // a warp-wide load: every lane, converged
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// The first n_ok (<= 16) of 16 values of one row: vector accesses when whole and aligned.
DF_DEVICE void st_row16(float* dst, const float (&v)[16], int n_ok) {
  if (n_ok >= 16 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < n_ok) dst[j] = v[j];
  }
}
DF_DEVICE void ld_row16(const float* src, float (&v)[16], int n_ok) {
  if (n_ok >= 16 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(src) + q);
      v[4 * q] = x.x;
      v[4 * q + 1] = x.y;
      v[4 * q + 2] = x.z;
      v[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = j < n_ok ? __ldcg(src + j) : 0.f;
  }
}
// The 16-bit hi/lo pair of 16 values of one row (the next projection's input).
DF_DEVICE void st_pair16(uint16_t* hi, uint16_t* lo, const float (&v)[16], bool f16, int n_ok) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) split_pair16x2(v[2 * e], v[2 * e + 1], f16, h[e], l[e]);
  if (n_ok >= 16 && ((reinterpret_cast<uintptr_t>(hi) | reinterpret_cast<uintptr_t>(lo)) & 15) == 0) {
    reinterpret_cast<uint4*>(hi)[0] = make_uint4(h[0], h[1], h[2], h[3]);
    reinterpret_cast<uint4*>(hi)[1] = make_uint4(h[4], h[5], h[6], h[7]);
    reinterpret_cast<uint4*>(lo)[0] = make_uint4(l[0], l[1], l[2], l[3]);
    reinterpret_cast<uint4*>(lo)[1] = make_uint4(l[4], l[5], l[6], l[7]);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < n_ok) {
        hi[j] = (uint16_t)(h[j >> 1] >> (16 * (j & 1)));
        lo[j] = (uint16_t)(l[j >> 1] >> (16 * (j & 1)));
      }
  }
}

// 1 / rms of one activation row from the previous kernel's per-tile sums of
// squares (summed in tile order).
DF_DEVICE float row_inv_rms(const GemmParams& p, int row) {
  float s = 0.f;
  int q = 0;
  for (; q + 8 <= p.n_ss; q += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcg(p.ss + (size_t)(q + u) * p.ss_ld + row);
#pragma unroll
    for (int u = 0; u < 8; ++u) s += v[u];
  }
  for (; q < p.n_ss; ++q) s += __ldcg(p.ss + (size_t)q * p.ss_ld + row);
  return 1.f / sqrtf(s / (float)p.rms_len + p.eps);
}

// The epilogue of one 128-column n-tile straight from tensor memory: each
// thread owns one activation row and 64 of the tile's columns, in one of two
// layouts - "plain" (warp half h: columns 64h .. 64h + 63) or "paired" (32h ..
// 32h + 31 and 64 + 32h .. 64 + 32h + 31: a SwiGLU gate column with its up
// column, or a rope pair of a 128-dim head).  Per-column scales and norm
// weights sit in the warp's scratch (wscr: [64] scales, [64] norm weights, in
// the thread's column order); row sums and argmax partials that span both
// halves are exchanged through xch ([2 parity][2 halves][128 rows]) at named
// barrier 3 + quadrant (the quadrant's two warps).  Outputs other than the
// residual stream go through the warp's staging tile stg (32 rows x 16
// columns, each row's columns rotated by row / 2 so that both the row-per-lane
// and the column-per-lane accesses are free of bank conflicts): a warp
// instruction then writes two (fp32) or four (16-bit pairs) row segments
// instead of 32 rows.
DF_DEVICE void epi_direct(const GemmParams& p, uint32_t tacc, int nt, int mt, int row, float inv,
                          int quad, int half, int lane, float* wscr, float2* xch, float* stg, int& n_xch,
                          int* s_flag) {
  const int epi = p.epi;
  const bool qkv = epi == EPI_QKV, paired = epi == EPI_SWIGLU || (qkv && p.hd == 128);
  const bool rok = row < p.M;
  const int rowbase = row - lane;   // the quadrant's first row
  auto col = [&](int c) { return paired ? (c < 32 ? 32 * half + c : 64 + 32 * half + c - 32) : 64 * half + c; };
  // head of this thread's columns (q/k/v): its first output column and kind
  const int n0h = nt * kTileRows + (paired ? 0 : 64 * half);
  const int kind = !qkv ? 0 : (n0h < p.qd ? 0 : (n0h < p.qd + p.kvd ? 1 : 2));
  __syncwarp();  // the previous tile's reads of the scratch are done
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int c = lane + 32 * e, cc = col(c);
    const float* sc = nullptr;
    const uint8_t* r = map_row(p, nt, cc, 1, &sc);
    wscr[c] = r ? (sc ? *sc : 1.f) : 0.f;
    float nw = 0.f;
    const int n = nt * kTileRows + cc;
    if (epi == EPI_RESID_SS && p.pair_hi && n < p.N) nw = load_dense(p.pair_norm, p.norm_bf16, n);
    if (qkv && kind != 2) nw = load_dense(kind == 0 ? p.q_norm : p.k_norm, p.norm_bf16, n - n0h);
    wscr[64 + c] = nw;
  }
  __syncwarp();
  const int xrow = quad * 32 + lane;
  float2* xb = xch + (size_t)(n_xch & 1) * 2 * 128;
  auto exchange = [&](float2 mine) {   // -> the other half's value for this row
    xb[half * 128 + xrow] = mine;
    __syncwarp();
    asm volatile("bar.sync %0, 64;" ::"r"(3 + quad) : "memory");
    ++n_xch;
    return xb[(half ^ 1) * 128 + xrow];
  };
  // staging tile: element (r, c) of the 32 x 16 chunk
  auto at = [&](int r, int c) { return r * 16 + ((c + (r >> 1)) & 15); };
  auto stage = [&](const float (&v)[16]) {
    __syncwarp();   // the previous chunk's reads are done
#pragma unroll
    for (int j = 0; j < 16; ++j) stg[at(lane, j)] = v[j];
    __syncwarp();
  };
  // columns [n0, n0 + 16) of the quadrant's rows at base + r * ld, below n_end
  auto store_t = [&](float* base, size_t ld, int n0, int n_end) {
#pragma unroll 4
    for (int it = 0; it < 16; ++it) {
      const int rr = 2 * it + (lane >> 4), c = lane & 15, r = rowbase + rr, n = n0 + c;
      if (r < p.M && n < n_end) base[(size_t)r * ld + n] = stg[at(rr, c)];
    }
  };
  // the 16-bit hi/lo pair of the staged chunk (times nw[c], if given)
  auto store_pair_t = [&](uint16_t* hi, uint16_t* lo, size_t ld, int n0, int n_end, const float* nw) {
    const bool f16 = p.pair_f16 != 0, even = (ld & 1) == 0;
#pragma unroll 4
    for (int it = 0; it < 8; ++it) {
      const int rr = 4 * it + (lane >> 3), c = 2 * (lane & 7), r = rowbase + rr, n = n0 + c;
      const float a = stg[at(rr, c)] * (nw ? nw[c] : 1.f), b = stg[at(rr, c + 1)] * (nw ? nw[c + 1] : 1.f);
      uint32_t h, l;
      split_pair16x2(a, b, f16, h, l);
      if (r >= p.M || n >= n_end) continue;
      const size_t o = (size_t)r * ld + n;
      if (even && n + 1 < n_end) {
        *reinterpret_cast<uint32_t*>(hi + o) = h;
        *reinterpret_cast<uint32_t*>(lo + o) = l;
      } else {
        hi[o] = (uint16_t)(h & 0xffffu);
        lo[o] = (uint16_t)(l & 0xffffu);
        if (n + 1 < n_end) {
          hi[o + 1] = (uint16_t)(h >> 16);
          lo[o + 1] = (uint16_t)(l >> 16);
        }
      }
    }
  };

  if (epi == EPI_SWIGLU) {
    const int F = p.seg[0].rows;
#pragma unroll 1
    for (int s = 0; s < 2; ++s) {
      float g[16], u[16];
      tmem_ld16(tacc + 32 * half + 16 * s, g);
      tmem_ld16(tacc + 64 + 32 * half + 16 * s, u);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float gv = g[j] * inv * wscr[16 * s + j];
        const float uv = u[j] * inv * wscr[32 + 16 * s + j];
        g[j] = gv / (1.f + expf(-gv)) * uv;
      }
      const int f0 = nt * (kTileRows / 2) + 32 * half + 16 * s;
      stage(g);
      if (p.out) store_t(p.out, p.ldo, f0, F);
      if (p.pair_hi) store_pair_t(p.pair_hi, p.pair_lo, p.pair_ld, f0, F, nullptr);
    }
    return;
  }

  if (qkv) {
    const int hd = p.hd, hh = hd / 2;
    const int d1 = paired ? 32 * half : 0;   // dims d1 + j (x1) and d1 + hh + j (x2), j < 32
    const int d_end = n0h < p.N ? hd : 0;   // no dims of a head past N
    float inv_h = 1.f;
    if (kind != 2) {
      float ss = 0.f;
#pragma unroll 1
      for (int s = 0; s < 2; ++s) {
        float a[16], b[16];
        tmem_ld16(tacc + col(16 * s), a);
        tmem_ld16(tacc + col(32 + 16 * s), b);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float x1 = a[j] * inv * wscr[16 * s + j], x2 = b[j] * inv * wscr[32 + 16 * s + j];
          ss += x1 * x1 + x2 * x2;
        }
      }
      if (paired) {
        const float o = exchange(make_float2(ss, 0.f)).x;
        ss = half == 0 ? ss + o : o + ss;   // the same order in both halves
      }
      inv_h = 1.f / sqrtf(ss / (float)hd + p.eps);
    }
    float* base = kind == 0 ? p.out + n0h : kind == 1 ? p.kblk + (n0h - p.qd) : p.vblk + (n0h - p.qd - p.kvd);
    const size_t ld = kind == 0 ? p.qd : p.kvd;
#pragma unroll 1
    for (int s = 0; s < 2; ++s) {
      float a[16], b[16];
      tmem_ld16(tacc + col(16 * s), a);
      tmem_ld16(tacc + col(32 + 16 * s), b);
      const int d = d1 + 16 * s;
      if (kind != 2) {
        const float4* cs4 = reinterpret_cast<const float4*>(p.rope_cs + (size_t)(rok ? row : 0) * hh + d);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 cs = __ldg(cs4 + q);   // (cos, sin) of dims d + 2q, d + 2q + 1
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = 2 * q + e;
            const float c = e ? cs.z : cs.x, sn = e ? cs.w : cs.y;
            const float x1 = a[j] * inv * wscr[16 * s + j], x2 = b[j] * inv * wscr[32 + 16 * s + j];
            const float u = x1 * inv_h * wscr[64 + 16 * s + j];
            const float w = x2 * inv_h * wscr[96 + 16 * s + j];
            a[j] = u * c - w * sn;
            b[j] = w * c + u * sn;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          a[j] = a[j] * inv * wscr[16 * s + j];
          b[j] = b[j] * inv * wscr[32 + 16 * s + j];
        }
      }
      stage(a);
      store_t(base, ld, d, d_end);
      stage(b);
      store_t(base, ld, d + hh, d_end);
    }
    return;
  }

  // rows: store, store + sums of squares, residual + sums of squares + pair, logits
  const bool resid = epi == EPI_RESID_SS, logits = epi == EPI_LOGITS;
  const bool ssk = epi == EPI_STORE_SS || resid;
  float ss = 0.f, bv = -CUDART_INF_F;
  int bi = 0x7fffffff;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    float v[16], res[16];
    tmem_ld16(tacc + 64 * half + 16 * s, v);
    const int n0 = nt * kTileRows + 64 * half + 16 * s;
    const int n_ok = rok ? max(0, min(16, p.N - n0)) : 0;
    if (resid && n_ok > 0)
      ld_row16(p.out + (size_t)row * p.ldo + n0, res, n_ok);
    else
#pragma unroll
      for (int j = 0; j < 16; ++j) res[j] = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float y = v[j] * inv * wscr[16 * s + j];
      if (j < n_ok) {
        y += res[j];
        if (logits) argmax_merge(bv, bi, y, n0 + j);
      } else {
        y = logits ? -CUDART_INF_F : 0.f;
      }
      v[j] = y;
      ss += y * y;
    }
    if (resid) {
      // one tile per CTA at these shapes: the epilogue is exposed, and per-row
      // vector accesses beat the staging round trip
      if (n_ok > 0) {
        st_row16(p.out + (size_t)row * p.ldo + n0, v, n_ok);
        if (p.pair_hi) {
#pragma unroll
          for (int j = 0; j < 16; ++j) res[j] = v[j] * wscr[64 + 16 * s + j];
          st_pair16(p.pair_hi + (size_t)row * p.pair_ld + n0, p.pair_lo + (size_t)row * p.pair_ld + n0, res,
                    p.pair_f16 != 0, n_ok);
        }
      }
    } else {
      stage(v);
      if (p.out) store_t(p.out, p.ldo, n0, p.N);
    }
  }
  if (ssk) {
    const float o = exchange(make_float2(ss, 0.f)).x;
    if (half == 0 && rok) p.ss_out[(size_t)nt * p.ss_out_ld + row] = ss + o;
  }
  if (logits) {
    const float2 o = exchange(make_float2(bv, __int_as_float(bi)));
    if (half == 0 && rok) {
      argmax_merge(bv, bi, o.x, __float_as_int(o.y));
      p.am_part[(size_t)nt * p.M + row] = make_float2(bv, __int_as_float(bi));
    }
    argmax_ticket(p, 8 * mt, min(8, p.n_mb - 8 * mt), s_flag);
  }
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
  constexpr int kS = Lt::kS;
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
      // the WR weight rows of item t in 32-row boxes: segment map and row
      auto tile_boxes = [&](int t, int* maps, int* rows) {
        const int wt2 = t / m_tiles;
#pragma unroll
        for (int q = 0; q < WR / 32; ++q) {
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
      };
      int maps[WR / 32], rows[WR / 32], nmaps[WR / 32], nrows[WR / 32];
      for (int t = blockIdx.x; t < n_items && !s_abort; t += G) {
        const int mt = t % m_tiles;
        tile_boxes(t, maps, rows);
        const bool next = t + G < n_items;
        if (next) tile_boxes(t + G, nmaps, nrows);
        for (int k = 0; k < nk; ++k, ++it) {
          // the weights kPf chunks ahead (this item's, or the next one's) into L2:
          // the box load then waits on L2 rather than on DRAM
          const bool cur = k + kPf < nk;
          const int kk = cur ? k + kPf : k + kPf - nk;
          if (kPf > 0 && (cur || (next && kk < nk))) {
#pragma unroll
            for (int q = 0; q < WR / 32; ++q)
              tma_prefetch2d(&p.tm_w[cur ? maps[q] : nmaps[q]], kk * 64, cur ? rows[q] : nrows[q]);
          }
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
    // straight from tensor memory where the epilogue's columns fit one thread
    // per row; injection and q/k/v heads of other widths take the staged path
    const bool direct = p.epi == EPI_SWIGLU || p.epi == EPI_RESID_SS || p.epi == EPI_STORE_SS ||
                        p.epi == EPI_STORE || p.epi == EPI_LOGITS ||
                        (p.epi == EPI_QKV && (p.hd == 64 || p.hd == 128));
    float* wscr = blk + warp * 128;                              // 8 x 128 floats
    float2* xch = reinterpret_cast<float2*>(blk + 8 * 128);     // 2 x 2 x 128 float2
    float* stg = blk + 16 * 128 + warp * 512;                   // 8 x 512 floats (into acc_s)
    static_assert((16 * 128 + 8 * 512) * 4 <= kOffInv - kOffBlk, "epilogue scratch");
    int n_xch = 0;
    int i = 0;
    for (int t = blockIdx.x; t < n_items; t += G, ++i) {
      const int mt = t % m_tiles, wt2 = t / m_tiles;
      const int buf = i & 1;
      // this lane's row and its 1 / rms, before the wait (overlaps the MMAs)
      const int row = mt * 128 + quad * 32 + lane;
      float inv = 1.f;
      if (direct && p.row_scale && row < p.M) inv = row_inv_rms(p, row);
      const bool ok = s_abort || bar_wait(&accf[buf], (uint32_t)((i >> 1) & 1));
      if (!ok && lane == 0) atomicOr(p.status, 0x4u);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      for (int sub = 0; direct && sub < kNsub; ++sub) {
        const int nt = kNsub * wt2 + sub;
        if (nt >= p.n_tiles) break;
        epi_direct(p, tmem + buf * kAccCols + ((uint32_t)(quad * 32) << 16) + sub * 128, nt, mt, row, inv,
                   quad, half, lane, wscr, xch, stg, n_xch, &s_flag);
      }
      for (int sub = 0; !direct && sub < kNsub; ++sub) {
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

size_t gemm_umma_smem_bytes() {
  return umma::L<256>::kSmem > umma::L<128>::kSmem ? umma::L<256>::kSmem : umma::L<128>::kSmem;
}

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
// give every SM a tile, else 128-row tiles for more parallelism.
cudaError_t launch_gemm_umma(int wt, const GemmParams& p, cudaStream_t st) {
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (n_sm <= 0) n_sm = 1;
  }
  const bool wide = (p.M + 127) / 128 * ((p.n_tiles + 1) / 2) >= n_sm;
  if (wt == W_BF16) return wide ? launch_umma_t<W_BF16, 256>(p, n_sm, st) : launch_umma_t<W_BF16, 128>(p, n_sm, st);
  if (wt == W_FP8) return wide ? launch_umma_t<W_FP8, 256>(p, n_sm, st) : launch_umma_t<W_FP8, 128>(p, n_sm, st);
  return cudaErrorInvalidValue;
}

}  // namespace dflash
