// dflash_encode_noalloc: the encode of dflash_encode for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside an
// allocator-free runtime, a host that has handed every byte of device memory to
// a pool it does not let callers carve from, or a plug-in that may only touch
// the buffers it is given.  dflash_create needs caller-allocated ring and
// scratch areas, so such callers cannot build a handle.  This entry point needs
// neither: the intermediate memory of the encode (split-K partial tiles, their
// tickets, per-tile sums of squares) lives in one file-scope __device__ array
// that every GPU loading this library holds until the process exits.  The
// caller passes only the weights, the features and the output buffer; the
// un-normalised projection is written into that output and normalised in place.
#include "../../include/dflash.h"
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <cstring>
#include <mutex>

using namespace dflash;

namespace {

constexpr size_t kScratchBytes = 8u << 20;          // 8 MiB per device
constexpr int kNaGrid = 152 * 2;                    // projection CTAs (one resident wave)
constexpr int kNaXk = kGemmXkMax;                   // activation stage width (shared limit)
constexpr size_t kCounterBytes = 64u << 10;         // tickets: 16384 ints
constexpr size_t kPartialBytes = (size_t)2 * kNaGrid * 16 * kTileRows * sizeof(float);
constexpr size_t kSsBytes = kScratchBytes - kCounterBytes - kPartialBytes;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device

// Once per device, with that device current: look up the device address of the
// array (the host-side symbol is only a stand-in, not a device address) and
// raise the projection kernels' shared-memory limit.
cudaError_t setup(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = configure_gemm(kNaXk);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_ptr[dev]);
  return cudaSuccess;
}

}  // namespace

extern "C" DFLASH_API int dflash_encode_noalloc(const dflash_config* cfg, const void* fc,
                                                const void* hidden_norm, const void* feats,
                                                int32_t T, float* H_t, void* stream) {
  if (!cfg || T < 0) return DFLASH_ERR_INVALID_ARG;
  if (cfg->n_embd < 1 || cfg->n_target_layers < 1 || cfg->target_embd < 1 || !(cfg->eps >= 0.f))
    return DFLASH_ERR_INVALID_ARG;
  if (cfg->dense_dtype != DFLASH_DTYPE_F32 && cfg->dense_dtype != DFLASH_DTYPE_BF16)
    return DFLASH_ERR_UNSUPPORTED;
  const int d = cfg->n_embd, fdim = cfg->n_target_layers * cfg->target_embd;
  if (d % 32 || fdim % 32) return DFLASH_ERR_UNSUPPORTED;
  if (T == 0) return DFLASH_OK;
  auto misaligned = [](const void* p) { return !p || (reinterpret_cast<uintptr_t>(p) & 15u); };
  if (misaligned(fc) || misaligned(hidden_norm) || misaligned(feats) || misaligned(H_t))
    return DFLASH_ERR_INVALID_ARG;
  const int n_tiles = (d + kTileRows - 1) / kTileRows, n_mb = (T + 15) / 16;
  // sizes beyond the static array: tickets (one per tile x 16-row block) and the
  // per-tile sums of squares of every row
  if ((size_t)n_tiles * n_mb * sizeof(int) > kCounterBytes ||
      (size_t)n_tiles * T * sizeof(float) > kSsBytes)
    return DFLASH_ERR_TOO_MANY_ROWS;

  // the runtime's last-error slot is shared with all CUDA work of the process:
  // an error left there by earlier work is not this call's
  (void)cudaGetLastError();
  unsigned char* base = nullptr;
  if (setup(&base) != cudaSuccess) return DFLASH_ERR_CUDA;
  int* counters = reinterpret_cast<int*>(base);
  float* partial = reinterpret_cast<float*>(base + kCounterBytes);
  float* ss = reinterpret_cast<float*>(base + kCounterBytes + kPartialBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the last call's contents: tickets must start at zero
  if (cudaMemsetAsync(counters, 0, (size_t)n_tiles * n_mb * sizeof(int), st) != cudaSuccess)
    return DFLASH_ERR_CUDA;

  const int dense_bf16 = cfg->dense_dtype == DFLASH_DTYPE_BF16;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.x = feats;
  p.x_mode = dense_bf16 ? X_BF16 : X_F32;
  p.ldx = fdim;
  p.M = T;
  p.K = fdim;
  p.eps = cfg->eps;
  p.norm_bf16 = dense_bf16;
  p.seg[0] = {fc, nullptr, 0, d};
  p.nseg = 1;
  p.N = d;
  p.map = MAP_SEGMENTS;
  p.n_tiles = n_tiles;
  p.n_mb = n_mb;
  p.cpt = fdim / 32;
  p.grid = (int)std::min<long long>(kNaGrid, (long long)n_tiles * n_mb * p.cpt);
  p.xk = std::min(fdim, kNaXk);
  p.partial = partial;
  p.counters = counters;
  p.epi = EPI_STORE_SS;
  p.out = H_t;          // un-normalised projection, normalised in place below
  p.ldo = d;
  p.ss_out = ss;
  p.ss_out_ld = T;
  if (launch_gemm(dense_bf16 ? W_BF16 : W_F32, p, st) != cudaSuccess) return DFLASH_ERR_CUDA;
  if (launch_rms_apply(H_t, ss, n_tiles, T, T, d, hidden_norm, dense_bf16, cfg->eps, H_t, st) !=
      cudaSuccess)
    return DFLASH_ERR_CUDA;
  return DFLASH_OK;
}
