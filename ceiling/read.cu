// Plain streaming read of a device buffer, for measurement: what one kernel
// launch reaches when it only moves bytes from HBM into the SMs, with no
// decode or arithmetic.  It is timed beside each weight product on a buffer
// of the same size, as that launch size's read ceiling.
//
// Each warp takes a contiguous range of chunks and streams them through a
// ring of `stages` shared-memory buffers filled by 1-D bulk copies
// (cp.async.bulk, completed on an mbarrier).  Every 16-byte word is folded
// into an XOR checksum, so no byte can be skipped; the warps' checksums are
// XORed into sink[0].  Waits are bounded: a wait that gives up sets sink[1]
// to 1, lets the copies in flight land and returns.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!try_wait(bar, parity))
    if (clock64() - t0 > (1ll << 32)) return false;
  return true;
}

__global__ void read_kernel(const uint8_t* __restrict__ src, long long bytes, int chunk, int stages,
                            long long wact, unsigned int* sink) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpc = blockDim.x >> 5;
  const long long wg = (long long)blockIdx.x * wpc + warp;
  if (wg >= wact) return;
  uint8_t* ring = smem + (size_t)warp * stages * chunk;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)wpc * stages * chunk) + warp * stages;
  const long long nch = (bytes + chunk - 1) / chunk;
  const long long c0 = nch * wg / wact, c1 = nch * (wg + 1) / wact;
  const int n = (int)(c1 - c0);
  if (lane == 0) {
    for (int i = 0; i < stages; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&bars[i])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  auto size_of = [&](long long c) { return (uint32_t)(c == nch - 1 ? bytes - c * chunk : chunk); };
  auto issue = [&](int i) {
    if (lane == 0) {
      const long long c = c0 + i;
      const int st = i % stages;
      const uint32_t bar = sa(&bars[st]), sz = size_of(c);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(sz) : "memory");
      asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       sa(ring + (size_t)st * chunk)),
                   "l"(src + c * chunk), "r"(sz), "r"(bar)
                   : "memory");
    }
  };
  int issued = 0;
  for (; issued < stages && issued < n; ++issued) issue(issued);
  uint32_t x = 0;
  bool ok = true;
  int i = 0;
  for (; i < n; ++i) {
    const int st = i % stages;
    if (!wait_bounded(sa(&bars[st]), (uint32_t)((i / stages) & 1))) {
      ok = false;
      break;
    }
    const uint4* w = reinterpret_cast<const uint4*>(ring + (size_t)st * chunk);
    const uint32_t words = size_of(c0 + i) / 16;
    for (uint32_t k = lane; k < words; k += 32) {
      const uint4 v = w[k];
      x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (issued < n) issue(issued++);
  }
  if (!ok) {
    if (lane == 0) atomicExch(&sink[1], 1u);
    for (; i < issued; ++i) (void)wait_bounded(sa(&bars[i % stages]), (uint32_t)((i / stages) & 1));
    return;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, o);
  if (lane == 0) atomicXor(&sink[0], x);
}

}  // namespace

extern "C" {

// Shared memory of one CTA.
size_t readceil_smem(int chunk, int warps, int stages) {
  return (size_t)warps * stages * chunk + (size_t)warps * stages * 8;
}

// Allows the kernel up to `max_smem` bytes of dynamic shared memory; call once
// before launching (and before any stream capture).  Returns a cudaError_t value.
int readceil_prepare(int max_smem) {
  return (int)cudaFuncSetAttribute(read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

// Reads `bytes` bytes at `src` (device, 16-byte aligned, bytes a multiple of
// 16) in chunks of `chunk` bytes (a multiple of 512), `warps` warps per CTA,
// up to `ctas` CTAs, `stages` buffers per warp; XORs every 32-bit word into
// sink[0] (device, two words; sink[1] is set to 1 if a wait gave up).
// readceil_prepare must have allowed the CTA's shared memory.  Returns a
// cudaError_t value.
int readceil_launch(const void* src, long long bytes, int chunk, int warps, int ctas, int stages, unsigned int* sink,
                    void* stream) {
  if (bytes <= 0 || bytes % 16 != 0 || chunk <= 0 || chunk % 512 != 0 || warps < 1 || warps > 32 || ctas < 1 ||
      stages < 1 || (reinterpret_cast<uintptr_t>(src) & 15u) != 0)
    return (int)cudaErrorInvalidValue;
  const size_t smem = readceil_smem(chunk, warps, stages);
  const long long nch = (bytes + chunk - 1) / chunk;
  const long long wmax = (long long)ctas * warps;
  const long long wact = nch < wmax ? nch : wmax;
  const int grid = (int)((wact + warps - 1) / warps);
  read_kernel<<<grid, warps * 32, smem, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint8_t*>(src), bytes,
                                                                             chunk, stages, wact, sink);
  return (int)cudaGetLastError();
}

}  // extern "C"
