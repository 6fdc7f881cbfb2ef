// rocmfp4_gemm_noalloc: the small-batch / GEMV product for callers that must
// not allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the
// product: an inference engine that hands all device memory to its own pool
// at start-up (an allocation behind its back could fail or fragment the
// memory it planned), a host with a real-time or certification rule against
// allocating after initialisation (allocation time is unbounded), or a
// plug-in loaded into a process whose allocator it must not touch.  The
// regular entry points allocate a per-device workspace on first use; this one
// never does.  Its scratch -- the split-tile partial sums, their hand-off
// counters and the error word of the streaming kernel -- lives in the
// file-scope array below, which every GPU that loads the library holds until
// the process exits.
//
// The format definition has no counterpart to this entry point: it is a
// deployment convenience of this library.
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/rocmfp4.h"
#include "kernels.h"

namespace {

using namespace rocmfp4;

// Scratch capacity: partial-sum records for at most kMaxWarps warps (two
// records of kStreamTileRows x 8 floats each), one counter per warp, one
// error word.
constexpr int kMaxWarps = 1024;
constexpr size_t kRecordFloats = (size_t)kStreamTileRows * 8;
constexpr size_t kRecordsBytes = sizeof(float) * kRecordFloats * 2 * kMaxWarps;    // 2 MiB
constexpr size_t kCountersBytes = sizeof(uint32_t) * kMaxWarps;                    // 4 KiB
constexpr size_t kScratchBytes = kRecordsBytes + kCountersBytes + 256;            // + error word

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct NoallocDevice {
  bool ready = false;
  int sms = 0;
  int occ[2][2][4] = {};  // streaming kernel CTAs per SM [variant][act][log2 mb]
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
NoallocDevice g_dev[kMaxDevices];

rocmfp4_status fail(rocmfp4_status st, const std::string& m) {
  set_last_error(m);  // reported by rocmfp4_last_error()
  return st;
}

rocmfp4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ROCMFP4_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// One-time set-up of the current device: the array's device address, kernel
// attributes, occupancy, and zeroed counters / error word.  No allocation.
rocmfp4_status setup(NoallocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ROCMFP4_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  NoallocDevice& d = g_dev[dev];
  if (!d.ready) {
    // In host code g_noalloc_scratch names a host-side stand-in; the kernel
    // needs the device address, fetched here with this device current.
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = stream_init_driver()) != cudaSuccess) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
    for (int v = 0; v < 2; ++v)
      for (int a = 0; a < 2; ++a)
        for (int lm = 0; lm < 4; ++lm) {
          if ((e = stream_prepare(v, a, 1 << lm)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
          if ((e = stream_occupancy(v, a, 1 << lm, &d.occ[v][a][lm])) != cudaSuccess)
            return cuda_fail(e, "occupancy");
          if (d.occ[v][a][lm] < 1) return fail(ROCMFP4_ERR_UNSUPPORTED, "streaming kernel does not fit");
        }
    // Counters and the error word must start at zero (the kernel returns the
    // counters to zero at the end of every completed call).
    unsigned char* s = static_cast<unsigned char*>(ptr);
    if ((e = cudaMemset(s + kRecordsBytes, 0, kCountersBytes + 256)) != cudaSuccess)
      return cuda_fail(e, "cudaMemset(scratch counters)");
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    d.scratch = s;
    d.ready = true;
  }
  *out = &d;
  return ROCMFP4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Reads (and clears) the error word of the array on the current device; a
// set word means a kernel gave up waiting and may have left split counters
// raised, so those are zeroed too.  A device without set-up has nothing to
// report.  Allocates nothing.
cudaError_t rocmfp4::noalloc_error_bits(cudaStream_t s, uint32_t* bits) {
  *bits = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev[dev].ready) scratch = g_dev[dev].scratch;
  }
  if (scratch == nullptr) return cudaSuccess;
  uint32_t v = 0;
  if ((e = cudaMemcpyAsync(&v, scratch + kRecordsBytes + kCountersBytes, sizeof(v), cudaMemcpyDeviceToHost, s)) !=
      cudaSuccess)
    return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  if (v != 0) {
    if ((e = cudaMemsetAsync(scratch + kRecordsBytes, 0, kCountersBytes + 256, s)) != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  }
  *bits = v;
  return cudaSuccess;
}

extern "C" rocmfp4_status rocmfp4_gemm_noalloc(const void* W, const void* X, float* Y, int64_t M, int64_t N,
                                               int64_t K, rocmfp4_variant variant, rocmfp4_act act,
                                               rocmfp4_stream_t stream) {
  if (variant != ROCMFP4_DUAL && variant != ROCMFP4_FAST) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown variant");
  if (act != ROCMFP4_ACT_F16 && act != ROCMFP4_ACT_BF16) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown activation type");
  if (M < 0 || N < 0 || K < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative size");
  if (K % 32 != 0) return fail(ROCMFP4_ERR_INVALID_ARG, "K must be a multiple of 32");
  if (M > 8)
    return fail(ROCMFP4_ERR_UNSUPPORTED,
                "rocmfp4_gemm_noalloc: M > 8 exceeds its fixed scratch (partial sums for at most 8 activation rows)");
  if (M == 0 || N == 0) return ROCMFP4_OK;
  if (!Y) return fail(ROCMFP4_ERR_INVALID_ARG, "Y is NULL");
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(Y, 0, sizeof(float) * M * N, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ROCMFP4_OK : cuda_fail(e, "cudaMemsetAsync");
  }
  if (!W || !X) return fail(ROCMFP4_ERR_INVALID_ARG, "NULL pointer");
  const int64_t ku = stream_weights_per_unit(variant);
  const int64_t units = (N + kStreamTileRows - 1) / kStreamTileRows * (K / ku);
  if (K % ku != 0 || !aligned16(W) || !aligned16(X) || units >= (int64_t(1) << 31))
    return fail(ROCMFP4_ERR_UNSUPPORTED,
                "rocmfp4_gemm_noalloc: needs K a multiple of 256 (dual) or 512 (single-scale), 16-byte aligned W "
                "and X, and fewer than 2^31 units");
  NoallocDevice* d = nullptr;
  rocmfp4_status st = setup(&d);
  if (st != ROCMFP4_OK) return st;

  const int mb = stream_mb_for((int)M);
  const int lm = mb == 1 ? 0 : mb == 2 ? 1 : mb == 4 ? 2 : 3;
  int64_t cap = (int64_t)d->sms * d->occ[variant][act][lm] * kStreamWarpsPerCta;
  if (cap > kMaxWarps) cap = kMaxWarps;  // the scratch holds records for kMaxWarps warps
  // the work split of rocmfp4_gemm_ex, within the array's capacity
  const int64_t tiles = (N + kStreamTileRows - 1) / kStreamTileRows;
  const int64_t wact = stream_warps(tiles, K / ku, ku * (variant == ROCMFP4_DUAL ? 18 : 17), M, cap);
  GemvArgs a{};
  a.W = static_cast<const uint8_t*>(W);
  a.X = static_cast<const uint16_t*>(X);
  a.Y = Y;
  a.N = N;
  a.K = K;
  a.row_bytes = K / 32 * (variant == ROCMFP4_DUAL ? 18 : 17);
  a.M = (int)M;
  a.nspans = K / ku;
  a.units = units;
  a.wact = wact;
  a.ws = reinterpret_cast<float*>(d->scratch);
  a.cnt = reinterpret_cast<uint32_t*>(d->scratch + kRecordsBytes);
  a.err = reinterpret_cast<uint32_t*>(d->scratch + kRecordsBytes + kCountersBytes);
  const int ctas = (int)((wact + kStreamWarpsPerCta - 1) / kStreamWarpsPerCta);
  a.deep = mb <= 2 && ctas <= 2 * d->sms ? 1 : 0;
  cudaError_t e = launch_gemv_stream(variant, act, a, ctas, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "streaming kernel launch");
  count_launch();
  return ROCMFP4_OK;
}
