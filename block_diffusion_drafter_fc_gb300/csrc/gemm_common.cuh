// Shared pieces of the two projection kernels: weight-row mapping, the
// stream-K schedule and fix-up, and the fused epilogues.  Everything here runs
// on the 256 "consumer" threads (threads 0..255) of a CTA and synchronises them
// with named barrier 1, so a kernel may add other warps (a TMA producer) that
// never enter these functions.
#pragma once

#include "common.cuh"
#include "internal.h"

#include <math_constants.h>

namespace dflash {

DF_DEVICE void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kGemmThreads) : "memory"); }

// Weight row `local` of `tile` -> its first byte (null when the row is past N).
DF_DEVICE const uint8_t* map_row(const GemmParams& p, int tile, int local, int esz,
                                 const float** scale) {
  int s = 0, r = 0;
  if (p.map == MAP_SWIGLU) {
    s = local < kTileRows / 2 ? 0 : 1;
    r = tile * (kTileRows / 2) + (local & (kTileRows / 2 - 1));
    if (r >= p.seg[s].rows) return nullptr;
  } else {
    const int vr = tile * kTileRows + local;
    if (vr >= p.N) return nullptr;
    while (s + 1 < p.nseg && vr >= p.seg[s + 1].row0) ++s;
    r = vr - p.seg[s].row0;
  }
  *scale = p.seg[s].scale ? p.seg[s].scale + r : nullptr;
  return reinterpret_cast<const uint8_t*>(p.seg[s].w) + (size_t)r * p.K * esz;
}

// Stream-K schedule: the work is n_items = n_tiles x n_mb output tiles (128
// weight rows x 16 activation rows), each cut into cpt chunks along k.  The
// grid is one resident wave; CTA b owns units [U b / G, U (b+1) / G) of the
// U = n_items * cpt units in item-major order, so every CTA streams the same
// number of weight bytes and there is no tail wave.  A tile finished inside one
// CTA goes straight to the epilogue; a tile shared by several CTAs is summed by
// the last of them (atomic ticket) in CTA order, which keeps results
// deterministic.  CTA c keeps at most two partial tiles: slot 2c for the tile
// its range starts inside, slot 2c + 1 for the tile its range ends inside.
DF_DEVICE long long owner_of(long long u, long long U, int G) { return ((u + 1) * G - 1) / U; }

// After a segment [c0, c1) of `item` has been accumulated into acc_s: publish
// it if the tile is shared and, for the last contributor, sum all partials in
// CTA order.  Returns true when this CTA must run the tile's epilogue.
DF_DEVICE bool segment_fixup(const GemmParams& p, float* acc_s, int item, int c0, int c1,
                             long long U, int G, int b, int* s_flag) {
  constexpr int kVec = 16 * kTileRows / 4;            // float4 per partial tile
  constexpr int kPer = kVec / kGemmThreads;           // float4 per thread
  const int tid = threadIdx.x;
  if (c0 == 0 && c1 == p.cpt) return true;
  const long long iu0 = (long long)item * p.cpt;
  const int first = (int)owner_of(iu0, U, G);
  const int last = (int)owner_of(iu0 + p.cpt - 1, U, G);
  float4* acc4 = reinterpret_cast<float4*>(acc_s);
  auto part_of = [&](int c) {
    const size_t sl = 2 * (size_t)c + (c == first ? 1 : 0);
    return reinterpret_cast<float4*>(p.partial + sl * (16 * kTileRows));
  };
  float4* mine = part_of(b);
#pragma unroll
  for (int k = 0; k < kPer; ++k) __stcg(mine + tid + k * kGemmThreads, acc4[tid + k * kGemmThreads]);
  // One thread takes the ticket with an acquire-release atomic after the CTA
  // barrier: the release publishes every thread's partial (the barrier orders
  // them before it), the acquire makes all earlier contributors' partials
  // visible to the winner, whose threads read them after the next barrier.
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
  // Sum the partials in CTA order; the loads of a batch of contributors are all
  // issued before the first add, so the fix-up costs about one L2 round trip
  // per batch rather than one per contributor.
  constexpr int kBatch = 4;
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

// Per-row 1 / rms of the 16 activation rows of block mb from the producer's
// per-tile sums of squares (16 threads per row, fixed-order tree).  Read from
// L2: in a projection chain another CTA of the same launch wrote them.
DF_DEVICE void compute_inv_rms(const GemmParams& p, float* inv_rms, int m0) {
  const int tid = threadIdx.x;
  const int m = tid >> 4, lq = tid & 15;
  float sum = 0.f;
  if (m0 + m < p.M)
    for (int q = lq; q < p.n_ss; q += 16) sum += __ldcg(p.ss + (size_t)q * p.ss_ld + m0 + m);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lq == 0) inv_rms[m] = 1.f / sqrtf(sum / (float)p.rms_len + p.eps);
}

// ------------------------------------------------------------------ epilogues

DF_DEVICE void argmax_ticket(const GemmParams& p, int mb0, int n_blocks, int* s_flag);

DF_DEVICE bool aligned16(const void* q) { return ((uintptr_t)q & 15) == 0; }

// Row epilogues of one finished 16 x 128 tile (store; residual add + the next
// projection's input pair + the rows' sums of squares; logits + per-row argmax).
// Thread t owns 8 consecutive columns of row t / 16: its loads and stores are
// 16-byte vectors (scalar at a ragged or unaligned edge), and a row's sum of
// squares or argmax is a shuffle reduction over the row's 16 threads.  With
// p.row_scale the accumulators are first multiplied by the row's 1 / rms.
DF_DEVICE void epilogue_rows(const GemmParams& p, const float* acc_s, const float* scale_s,
                             const float* inv_rms, int mb, int tile, int* s_flag) {
  const int tid = threadIdx.x, m = tid >> 4, c0 = (tid & 15) * 8;
  const int row = mb * 16 + m, n0 = tile * kTileRows + c0;
  const bool logits = p.epi == EPI_LOGITS, resid = p.epi == EPI_RESID_SS;
  const bool pair = resid && p.pair_hi != nullptr;
  const int nv = row < p.M ? max(0, min(8, p.N - n0)) : 0;   // this thread's valid columns
  float* o = p.out ? p.out + (size_t)row * p.ldo + n0 : nullptr;
  uint16_t* oh = pair ? p.pair_hi + (size_t)row * p.pair_ld + n0 : nullptr;
  uint16_t* ol = pair ? p.pair_lo + (size_t)row * p.pair_ld + n0 : nullptr;
  const char* nwp = pair ? static_cast<const char*>(p.pair_norm) + (size_t)n0 * (p.norm_bf16 ? 2 : 4)
                         : nullptr;
  const bool vec = nv == 8 && (!o || aligned16(o)) &&
                   (!pair || (aligned16(oh) && aligned16(ol) && aligned16(nwp)));
  // the residual and the next norm's weights, all loads first
  float res[8], nw[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) res[j] = nw[j] = 0.f;
  if (resid && vec) {
    const float4 r0 = __ldcg(reinterpret_cast<const float4*>(o));
    const float4 r1 = __ldcg(reinterpret_cast<const float4*>(o) + 1);
    res[0] = r0.x; res[1] = r0.y; res[2] = r0.z; res[3] = r0.w;
    res[4] = r1.x; res[5] = r1.y; res[6] = r1.z; res[7] = r1.w;
    if (pair && p.norm_bf16) {
      const uint4 w = *reinterpret_cast<const uint4*>(nwp);
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        nw[2 * j] = bf16_bits_to_f32((uint16_t)(wv[j] & 0xffffu));
        nw[2 * j + 1] = bf16_bits_to_f32((uint16_t)(wv[j] >> 16));
      }
    } else if (pair) {
      const float4 w0 = *reinterpret_cast<const float4*>(nwp);
      const float4 w1 = *(reinterpret_cast<const float4*>(nwp) + 1);
      nw[0] = w0.x; nw[1] = w0.y; nw[2] = w0.z; nw[3] = w0.w;
      nw[4] = w1.x; nw[5] = w1.y; nw[6] = w1.z; nw[7] = w1.w;
    }
  } else if (resid) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < nv) {
        res[j] = __ldcg(o + j);
        if (pair) nw[j] = load_dense(p.pair_norm, p.norm_bf16, n0 + j);
      }
  }
  const float inv = p.row_scale ? inv_rms[m] : 1.f;
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a = acc_s[m * kTileRows + c0 + j];
    if (p.row_scale) a *= inv;
    y[j] = a * scale_s[c0 + j];
    if (resid) y[j] += res[j];
    if (j >= nv) y[j] = 0.f;
  }
  if (vec) {
    if (o) {
      reinterpret_cast<float4*>(o)[0] = make_float4(y[0], y[1], y[2], y[3]);
      reinterpret_cast<float4*>(o)[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
    if (pair) {
      // the next projection's input: split(h * next norm weight)
      uint32_t h[4], l[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        split_pair16x2(y[2 * j] * nw[2 * j], y[2 * j + 1] * nw[2 * j + 1], p.pair_f16 != 0, h[j], l[j]);
      *reinterpret_cast<uint4*>(oh) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(ol) = make_uint4(l[0], l[1], l[2], l[3]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < nv) {
        if (o) o[j] = y[j];
        if (pair) {
          uint16_t zh, zl;
          split_pair16(y[j] * nw[j], p.pair_f16 != 0, zh, zl);
          oh[j] = zh;
          ol[j] = zl;
        }
      }
  }
  if (p.epi == EPI_STORE_SS || resid) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += y[j] * y[j];
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 15) == 0 && row < p.M) p.ss_out[(size_t)tile * p.ss_out_ld + row] = ss;
  }
  if (!logits) return;
  float v = -CUDART_INF_F;
  int idx = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < nv) argmax_merge(v, idx, y[j], n0 + j);
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, off);
    argmax_merge(v, idx, v2, i2);
  }
  if ((tid & 15) == 0 && row < p.M) p.am_part[(size_t)tile * p.M + row] = make_float2(v, __int_as_float(idx));
  argmax_ticket(p, mb, 1, s_flag);
}

// After a CTA has written the argmax partials of 16-row blocks mb0 ..
// mb0 + n_blocks - 1 (n_blocks <= 8) for one tile: take one ticket per block
// (acquire-release, as in segment_fixup; am_counter[mb] counts the block's
// finished tiles).  The CTA that takes a block's last ticket reduces the
// block's rows over the tiles (lowest index on ties) into its drafts and resets
// the block's counter, so the reductions spread over the CTAs.
DF_DEVICE void argmax_ticket(const GemmParams& p, int mb0, int n_blocks, int* s_flag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  csync();
  if (warp == 0) {
    bool won = false;
    if (lane < n_blocks) {
      int old;
      asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                   : "=r"(old)
                   : "l"(p.am_counter + mb0 + lane)
                   : "memory");
      won = old == p.n_tiles - 1;
      if (won) p.am_counter[mb0 + lane] = 0;   // every ticket of the block is taken
    }
    const unsigned mask = __ballot_sync(0xffffffffu, won);
    if (lane == 0) *s_flag = (int)mask;
  }
  csync();
  const unsigned mask = (unsigned)*s_flag;
  if (!mask) return;
  for (int k = warp; k < n_blocks * 16; k += kGemmThreads / 32) {
    const int bb = k >> 4, i = k & 15, row = (mb0 + bb) * 16 + i;
    if (!((mask >> bb) & 1u) || i == 0 || row >= p.M) continue;
    float v = -CUDART_INF_F;
    int idx = 0x7fffffff;
    for (int tt = lane; tt < p.n_tiles; tt += 32) {
      const float2 e = __ldcg(p.am_part + (size_t)tt * p.M + row);
      argmax_merge(v, idx, e.x, __float_as_int(e.y));
    }
    warp_argmax(v, idx);
    if (lane == 0) p.drafts[(row >> 4) * 15 + i - 1] = i < p.block_width ? idx : -1;
  }
}

// SwiGLU of one finished tile (gate rows 0..63, up rows 64..127): thread t
// owns 4 consecutive outputs of row t / 16 (8-byte pair stores, 16-byte output
// stores; scalar at a ragged or unaligned edge).
DF_DEVICE void epilogue_swiglu(const GemmParams& p, const float* acc_s, const float* scale_s,
                               const float* inv_rms, int mb, int tile) {
  constexpr int half = kTileRows / 2;
  const int tid = threadIdx.x, m = tid >> 4, j0 = (tid & 15) * 4;
  const int row = mb * 16 + m, f0 = tile * half + j0;
  const int nv = row < p.M ? max(0, min(4, p.seg[0].rows - f0)) : 0;
  if (nv == 0) return;
  const float inv = p.row_scale ? inv_rms[m] : 1.f;
  float a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float g = acc_s[m * kTileRows + j0 + j], u = acc_s[m * kTileRows + half + j0 + j];
    if (p.row_scale) {
      g *= inv;
      u *= inv;
    }
    const float gv = g * scale_s[j0 + j], uv = u * scale_s[half + j0 + j];
    a[j] = j < nv ? gv / (1.f + expf(-gv)) * uv : 0.f;
  }
  float* o = p.out ? p.out + (size_t)row * p.ldo + f0 : nullptr;
  uint16_t* oh = p.pair_hi ? p.pair_hi + (size_t)row * p.pair_ld + f0 : nullptr;
  uint16_t* ol = p.pair_hi ? p.pair_lo + (size_t)row * p.pair_ld + f0 : nullptr;
  const bool vec = nv == 4 && (!o || aligned16(o)) &&
                   (!oh || ((((uintptr_t)oh | (uintptr_t)ol) & 7) == 0));
  if (vec) {
    if (o) *reinterpret_cast<float4*>(o) = make_float4(a[0], a[1], a[2], a[3]);
    if (oh) {
      uint32_t h0, l0, h1, l1;
      split_pair16x2(a[0], a[1], p.pair_f16 != 0, h0, l0);
      split_pair16x2(a[2], a[3], p.pair_f16 != 0, h1, l1);
      *reinterpret_cast<uint2*>(oh) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(ol) = make_uint2(l0, l1);
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nv) {
      if (o) o[j] = a[j];
      if (oh) {
        uint16_t ah, al;
        split_pair16(a[j], p.pair_f16 != 0, ah, al);
        oh[j] = ah;
        ol[j] = al;
      }
    }
}

// Per-head RMSNorm + NEOX rope of q/k (raw v) for the block (EPI_QKV) or for
// injected context rows scattered into the ring (EPI_INJECT).  One half-warp per
// (row, head) item: lane l holds the per = hd / 32 consecutive elements
// [l per, (l + 1) per) of the head's first half and their rope partners in the
// second half, so the head's sum of squares is a 16-lane shuffle reduction and
// the q/k/v stores are vectors.  Every lane takes part in the shuffles; items
// past the tile's rows or columns are skipped only after them.
DF_DEVICE void epilogue_heads(const GemmParams& p, const float* acc_s, const float* scale_s,
                              const float* inv_rms, int mb, int tile) {
  const int lane = threadIdx.x & 31, l16 = lane & 15;
  const int hwi = (threadIdx.x >> 5) * 2 + (lane >> 4);   // half-warp 0..15
  const int hd = p.hd, half = hd >> 1, hpt = kTileRows / hd, per = half / 16;
  const int j0 = l16 * per;
  for (int item = hwi; item < 16 * hpt; item += 16) {
    const int m = item / hpt, hh = item - m * hpt;
    const int n0 = tile * kTileRows + hh * hd, row = mb * 16 + m;
    const bool live = n0 < p.N && row < p.M;
    int kind = 2, layer = 0, head = 0;
    const void* normw = nullptr;
    if (p.epi == EPI_QKV) {
      kind = n0 < p.qd ? 0 : (n0 < p.qd + p.kvd ? 1 : 2);
      normw = kind == 0 ? p.q_norm : p.k_norm;
    } else {
      layer = n0 / (2 * p.kvd);
      const int w = n0 - layer * 2 * p.kvd;
      kind = w < p.kvd ? 1 : 2;
      head = (w - (kind == 2 ? p.kvd : 0)) / hd;
      if (live) normw = p.k_norm_l[layer];
    }
    const bool rope = live && kind != 2;
    // the norm weights and the row's rope entries first: their loads overlap the
    // tile reads and the reduction
    float wa[4], wb[4];
    float2 cs[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      wa[q] = wb[q] = 0.f;
      cs[q] = make_float2(0.f, 0.f);
      if (rope && q < per) {
        wa[q] = load_dense(normw, p.norm_bf16, j0 + q);
        wb[q] = load_dense(normw, p.norm_bf16, j0 + q + half);
        cs[q] = p.rope_cs[(size_t)row * half + j0 + q];
      }
    }
    const float* src = acc_s + m * kTileRows + hh * hd;
    const float* sc = scale_s + hh * hd;
    const float rs = p.row_scale ? inv_rms[m] : 1.f;
    float x1[4], x2[4];
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x1[q] = x2[q] = 0.f;
      if (q < per) {
        const int j = j0 + q;
        float s1 = src[j], s2 = src[j + half];
        if (p.row_scale) {
          s1 *= rs;
          s2 *= rs;
        }
        x1[q] = s1 * sc[j];
        x2[q] = s2 * sc[j + half];
      }
      ss += x1[q] * x1[q] + x2[q] * x2[q];
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (!live) continue;
    if (kind != 2) {
      const float inv = 1.f / sqrtf(ss / (float)hd + p.eps);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = x1[q] * inv * wa[q];
        const float b = x2[q] * inv * wb[q];
        x1[q] = a * cs[q].x - b * cs[q].y;
        x2[q] = b * cs[q].x + a * cs[q].y;
      }
    }
    if (p.epi == EPI_QKV) {
      float* dst = kind == 0 ? p.out + (size_t)row * p.qd + n0
                 : kind == 1 ? p.kblk + (size_t)row * p.kvd + (n0 - p.qd)
                             : p.vblk + (size_t)row * p.kvd + (n0 - p.qd - p.kvd);
      if (per == 4 && aligned16(dst)) {
        reinterpret_cast<float4*>(dst + j0)[0] = make_float4(x1[0], x1[1], x1[2], x1[3]);
        reinterpret_cast<float4*>(dst + half + j0)[0] = make_float4(x2[0], x2[1], x2[2], x2[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < per) {
            dst[j0 + q] = x1[q];
            dst[j0 + q + half] = x2[q];
          }
      }
    } else {
      int sq = 0;
      if (p.rows_per_seq > 0) {
        sq = row / p.rows_per_seq;
        if (p.row_count && row - sq * p.rows_per_seq >= p.row_count[sq]) continue;
      }
      const int pos = p.pos[row];
      if (pos < 0) {
        if (l16 == 0) atomicOr(p.status, 0x2u);
        continue;
      }
      const int slot = pos % p.window;
      const size_t off =
          ((((size_t)layer * 2 + (kind == 2)) * p.n_head_kv + head) * p.window + slot) * hd;
      void* ring_base = static_cast<char*>(p.ring_seq) + (size_t)sq * p.ring_seq_stride;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q >= per) continue;
        const int j = j0 + q;
        if (p.ring_bf16) {
          uint16_t* d = reinterpret_cast<uint16_t*>(ring_base) + off;
          d[j] = f32_to_bf16_bits(x1[q]);
          d[j + half] = f32_to_bf16_bits(x2[q]);
        } else {
          float* d = reinterpret_cast<float*>(ring_base) + off;
          d[j] = x1[q];
          d[j + half] = x2[q];
        }
      }
    }
  }
}


// Run the fused epilogue of one finished 16 x 128 tile.  With p.row_scale each
// epilogue first multiplies the accumulators by their row's 1 / rms (RMSNorm
// applied after the projection: a per-row scalar commutes with the product).
DF_DEVICE void run_epilogue(const GemmParams& p, float* acc_s, const float* scale_s,
                            const float* inv_rms, int mb, int tile, int* s_flag) {
  switch (p.epi) {
    case EPI_SWIGLU:
      epilogue_swiglu(p, acc_s, scale_s, inv_rms, mb, tile);
      break;
    case EPI_QKV:
    case EPI_INJECT:
      epilogue_heads(p, acc_s, scale_s, inv_rms, mb, tile);
      break;
    default:
      epilogue_rows(p, acc_s, scale_s, inv_rms, mb, tile, s_flag);
      break;
  }
}

}  // namespace dflash
