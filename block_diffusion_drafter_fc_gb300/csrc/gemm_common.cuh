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

DF_DEVICE void epilogue_rows(const GemmParams& p, float* acc_s, const float* scale_s, int mb,
                             int tile, int* s_flag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = mb * 16;
  const bool logits = p.epi == EPI_LOGITS;
  constexpr int kPer = 16 * kTileRows / kGemmThreads;
  const bool resid = p.epi == EPI_RESID_SS;
  // the residual rows and next-norm weights this thread needs, all loads first
  float res[kPer], nw[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = tid + k * kGemmThreads;
    const int m = i / kTileRows, r = i - m * kTileRows;
    const int n = tile * kTileRows + r, row = m0 + m;
    const bool ok = n < p.N && row < p.M;
    res[k] = resid && ok ? __ldcg(p.out + (size_t)row * p.ldo + n) : 0.f;
    nw[k] = resid && ok && p.pair_hi ? load_dense(p.pair_norm, p.norm_bf16, n) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = tid + k * kGemmThreads;
    const int m = i / kTileRows, r = i - m * kTileRows;
    const int n = tile * kTileRows + r, row = m0 + m;
    float y = acc_s[i] * scale_s[r];
    if (n < p.N && row < p.M) {
      if (resid) {
        y += res[k];
        p.out[(size_t)row * p.ldo + n] = y;
        if (p.pair_hi) {
          // the next projection's input: split(h * next norm weight)
          uint16_t zh, zl;
          split_pair16(y * nw[k], p.pair_f16 != 0, zh, zl);
          p.pair_hi[(size_t)row * p.pair_ld + n] = zh;
          p.pair_lo[(size_t)row * p.pair_ld + n] = zl;
        }
      } else if (p.out) {
        p.out[(size_t)row * p.ldo + n] = y;
      }
    } else {
      y = logits ? -CUDART_INF_F : 0.f;
    }
    acc_s[i] = y;
  }
  csync();
  if (p.epi == EPI_STORE_SS || p.epi == EPI_RESID_SS) {
    for (int m = warp; m < 16; m += kGemmThreads / 32) {
      float s = 0.f;
      for (int r = lane; r < kTileRows; r += 32) s += acc_s[m * kTileRows + r] * acc_s[m * kTileRows + r];
      s = warp_sum(s);
      if (lane == 0 && m0 + m < p.M) p.ss_out[(size_t)tile * p.ss_out_ld + m0 + m] = s;
    }
  }
  if (!logits) return;
  for (int m = warp; m < 16; m += kGemmThreads / 32) {
    float v = -CUDART_INF_F;
    int idx = 0x7fffffff;
    for (int r = lane; r < kTileRows; r += 32) {
      const int n = tile * kTileRows + r;
      if (n < p.N) argmax_merge(v, idx, acc_s[m * kTileRows + r], n);
    }
    warp_argmax(v, idx);
    if (lane == 0 && m0 + m < p.M)
      p.am_part[(size_t)tile * p.M + m0 + m] = make_float2(v, __int_as_float(idx));
  }
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

DF_DEVICE void epilogue_swiglu(const GemmParams& p, const float* acc_s, const float* scale_s,
                               int mb, int tile) {
  const int half = kTileRows / 2, F = p.seg[0].rows;
  for (int i = threadIdx.x; i < 16 * half; i += kGemmThreads) {
    const int m = i / half, j = i - m * half;
    const int f = tile * half + j, row = mb * 16 + m;
    if (f >= F || row >= p.M) continue;
    const float gv = acc_s[m * kTileRows + j] * scale_s[j];
    const float uv = acc_s[m * kTileRows + half + j] * scale_s[half + j];
    const float a = gv / (1.f + expf(-gv)) * uv;
    if (p.out) p.out[(size_t)row * p.ldo + f] = a;
    if (p.pair_hi) {
      uint16_t ah, al;
      split_pair16(a, p.pair_f16 != 0, ah, al);
      p.pair_hi[(size_t)row * p.pair_ld + f] = ah;
      p.pair_lo[(size_t)row * p.pair_ld + f] = al;
    }
  }
}

// Per-head RMSNorm + NEOX rope of q/k (raw v) for the block (EPI_QKV) or for
// injected context rows scattered into the ring (EPI_INJECT).
DF_DEVICE void epilogue_heads(const GemmParams& p, const float* acc_s, const float* scale_s,
                              int mb, int tile) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hd = p.hd, half = hd >> 1, hpt = kTileRows / hd;
  for (int item = warp; item < 16 * hpt; item += kGemmThreads / 32) {
    const int m = item / hpt, hh = item - m * hpt;
    const int n0 = tile * kTileRows + hh * hd, row = mb * 16 + m;
    if (n0 >= p.N || row >= p.M) continue;
    int kind, layer = 0, head = 0;
    const void* normw;
    if (p.epi == EPI_QKV) {
      kind = n0 < p.qd ? 0 : (n0 < p.qd + p.kvd ? 1 : 2);
      normw = kind == 0 ? p.q_norm : p.k_norm;
    } else {
      layer = n0 / (2 * p.kvd);
      const int w = n0 - layer * 2 * p.kvd;
      kind = w < p.kvd ? 1 : 2;
      head = (w - (kind == 2 ? p.kvd : 0)) / hd;
      normw = p.k_norm_l[layer];
    }
    const float* src = acc_s + m * kTileRows + hh * hd;
    const float* sc = scale_s + hh * hd;
    float x1[4], x2[4];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = lane + 32 * u;
      x1[u] = j < half ? src[j] * sc[j] : 0.f;
      x2[u] = j < half ? src[j + half] * sc[j + half] : 0.f;
      ss += x1[u] * x1[u] + x2[u] * x2[u];
    }
    if (kind != 2) {
      ss = warp_sum(ss);
      const float inv = 1.f / sqrtf(ss / (float)hd + p.eps);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = lane + 32 * u;
        if (j >= half) continue;
        const float a = x1[u] * inv * load_dense(normw, p.norm_bf16, j);
        const float b = x2[u] * inv * load_dense(normw, p.norm_bf16, j + half);
        const float2 cs = p.rope_cs[(size_t)row * half + j];
        x1[u] = a * cs.x - b * cs.y;
        x2[u] = b * cs.x + a * cs.y;
      }
    }
    if (p.epi == EPI_QKV) {
      float* dst = kind == 0 ? p.out + (size_t)row * p.qd + n0
                 : kind == 1 ? p.kblk + (size_t)row * p.kvd + (n0 - p.qd)
                             : p.vblk + (size_t)row * p.kvd + (n0 - p.qd - p.kvd);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = lane + 32 * u;
        if (j < half) {
          dst[j] = x1[u];
          dst[j + half] = x2[u];
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
        if (lane == 0) atomicOr(p.status, 0x2u);
        continue;
      }
      const int slot = pos % p.window;
      const size_t off =
          ((((size_t)layer * 2 + (kind == 2)) * p.n_head_kv + head) * p.window + slot) * hd;
      void* ring_base = static_cast<char*>(p.ring_seq) + (size_t)sq * p.ring_seq_stride;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = lane + 32 * u;
        if (j >= half) continue;
        if (p.ring_bf16) {
          uint16_t* d = reinterpret_cast<uint16_t*>(ring_base) + off;
          d[j] = f32_to_bf16_bits(x1[u]);
          d[j + half] = f32_to_bf16_bits(x2[u]);
        } else {
          float* d = reinterpret_cast<float*>(ring_base) + off;
          d[j] = x1[u];
          d[j + half] = x2[u];
        }
      }
    }
  }
}


// Run the fused epilogue of one finished 16 x 128 tile.  With p.row_scale the
// tile rows are first multiplied by 1 / rms (RMSNorm applied after the
// projection: a per-row scalar commutes with the product).
DF_DEVICE void run_epilogue(const GemmParams& p, float* acc_s, const float* scale_s,
                            const float* inv_rms, int mb, int tile, int* s_flag) {
  if (p.row_scale) {
    for (int i = threadIdx.x; i < 16 * kTileRows; i += kGemmThreads) acc_s[i] *= inv_rms[i / kTileRows];
    csync();
  }
  switch (p.epi) {
    case EPI_SWIGLU:
      epilogue_swiglu(p, acc_s, scale_s, mb, tile);
      break;
    case EPI_QKV:
    case EPI_INJECT:
      epilogue_heads(p, acc_s, scale_s, mb, tile);
      break;
    default:
      epilogue_rows(p, acc_s, scale_s, mb, tile, s_flag);
      break;
  }
}

}  // namespace dflash
