// Elementwise ROCmFP4 kernels: dequantisation, scale validation, and the
// generic product used when a shape or pointer alignment does not fit the
// streaming kernel.  Decode follows "Feasibility Report: Porting ROCmFP4 to
// Atlas", section "What is ROCmFP4?" (Block Layout, Codebook10 Value Table,
// Scale Format), in plain fp32 arithmetic that is exact for every weight.
#include "common.cuh"
#include "kernels.h"

namespace rocmfp4 {
namespace {

// Codebook10[q] as an exact float; code 8 gives +0.
RF4_DEV float codebook10(uint32_t q) {
  const int m = (int)(q & 7u);
  const int v = m <= 4 ? m : 2 * m - 4;  // 0 1 2 3 4 6 8 10
  return (float)((q & 8u) ? -v : v);
}

RF4_DEV float act_to_f32(uint16_t bits, int act) {
  if (act == 0) return __half2float(__ushort_as_half(bits));
  return __uint_as_float((uint32_t)bits << 16);
}

// ---- dequant: one thread per 8 consecutive weights of one block half ------------
template <int V, int OUT, bool VEC>
__global__ void dequant_kernel(const uint8_t* __restrict__ W, void* __restrict__ out, int64_t nblocks) {
  constexpr int BB = Fmt<V>::BB;
  const int64_t nchunks = nblocks * 4;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < nchunks;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = g >> 2;
    const int qi = (int)(g & 3);
    const int h = qi >> 1, j0 = (qi & 1) * 8;
    const uint8_t* b = W + blk * BB;
    const float hs = halfscale_f32(__ldg(b + 16 + (V == 0 ? h : 0)));
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = __ldg(b + j0 + i);
      // + 0 turns the -0 of a negative code times a zero scale into +0
      v[i] = __fadd_rn(codebook10(h ? (byte >> 4) : (byte & 15u)) * hs, 0.0f);
    }
    const int64_t o = blk * 32 + 16 * h + j0;
    if constexpr (OUT == 0) {
      float* dst = static_cast<float*>(out) + o;
      if constexpr (VEC) {
        reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = v[i];
      }
    } else {
      uint16_t r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        r[i] = OUT == 1 ? __bfloat16_as_ushort(__float2bfloat16_rn(v[i])) : __half_as_ushort(__float2half_rn(v[i]));
      uint16_t* dst = static_cast<uint16_t*>(out) + o;
      if constexpr (VEC) {
        uint4 pk;
        pk.x = r[0] | ((uint32_t)r[1] << 16);
        pk.y = r[2] | ((uint32_t)r[3] << 16);
        pk.z = r[4] | ((uint32_t)r[5] << 16);
        pk.w = r[6] | ((uint32_t)r[7] << 16);
        *reinterpret_cast<uint4*>(dst) = pk;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = r[i];
      }
    }
  }
}

// ---- validate --------------------------------------------------------------------
template <int V>
__global__ void validate_kernel(const uint8_t* __restrict__ W, int64_t nblocks, unsigned long long* first) {
  constexpr int BB = Fmt<V>::BB;
  for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblocks;
       blk += (int64_t)gridDim.x * blockDim.x) {
    bool bad = __ldg(W + blk * BB + 16) >= 0x7Fu;
    if (V == 0) bad = bad || __ldg(W + blk * BB + 17) >= 0x7Fu;
    if (bad) atomicMin(first, (unsigned long long)blk);
  }
}

// ---- generic product: one warp per row, lanes over blocks -----------------------
template <int V>
__global__ void gemm_generic_kernel(const GenericArgs a, int act) {
  constexpr int BB = Fmt<V>::BB;
  const int lane = threadIdx.x & 31;
  const int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (n >= a.N) return;
  const int64_t nb = a.K / 32;
  const uint8_t* row = a.W + n * a.row_bytes;
  for (int64_t m0 = 0; m0 < a.M; m0 += 4) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t b = lane; b < nb; b += 32) {
      const uint8_t* blk = row + b * BB;
      const float hs0 = halfscale_f32(blk[16]);
      const float hs1 = V == 0 ? halfscale_f32(blk[17]) : hs0;
      for (int i = 0; i < 32; ++i) {
        const uint32_t byte = blk[i & 15];
        const float w = codebook10(i < 16 ? (byte & 15u) : (byte >> 4)) * (i < 16 ? hs0 : hs1);
#pragma unroll
        for (int mm = 0; mm < 4; ++mm)
          if (m0 + mm < a.M) s[mm] = fmaf(w, act_to_f32(a.X[(m0 + mm) * a.K + b * 32 + i], act), s[mm]);
      }
    }
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      float v = s[mm];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && m0 + mm < a.M) a.Y[(m0 + mm) * a.N + n] = v;
    }
  }
}

int grid_for(int64_t work, int threads) {
  int64_t g = (work + threads - 1) / threads;
  if (g > 152 * 32) g = 152 * 32;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_dequant(int variant, int out_dtype, const uint8_t* W, void* out, int64_t nblocks,
                           cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  const bool vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  const int threads = 256, grid = grid_for(nblocks * 4, threads);
#define RF4_DQ(V, O)                                                                        \
  do {                                                                                      \
    if (vec) dequant_kernel<V, O, true><<<grid, threads, 0, s>>>(W, out, nblocks);         \
    else dequant_kernel<V, O, false><<<grid, threads, 0, s>>>(W, out, nblocks);            \
  } while (0)
  if (variant == 0) {
    if (out_dtype == 0) RF4_DQ(0, 0); else if (out_dtype == 1) RF4_DQ(0, 1); else RF4_DQ(0, 2);
  } else {
    if (out_dtype == 0) RF4_DQ(1, 0); else if (out_dtype == 1) RF4_DQ(1, 1); else RF4_DQ(1, 2);
  }
#undef RF4_DQ
  return cudaGetLastError();
}

cudaError_t launch_validate(int variant, const uint8_t* W, int64_t nblocks, unsigned long long* first,
                            cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  const int threads = 256, grid = grid_for(nblocks, threads);
  if (variant == 0) validate_kernel<0><<<grid, threads, 0, s>>>(W, nblocks, first);
  else validate_kernel<1><<<grid, threads, 0, s>>>(W, nblocks, first);
  return cudaGetLastError();
}

cudaError_t launch_gemm_generic(int variant, int act, const GenericArgs& a, cudaStream_t s) {
  if (a.N == 0 || a.M == 0) return cudaSuccess;
  const int warps = 4;
  const int64_t grid = (a.N + warps - 1) / warps;
  if (variant == 0) gemm_generic_kernel<0><<<(unsigned)grid, warps * 32, 0, s>>>(a, act);
  else gemm_generic_kernel<1><<<(unsigned)grid, warps * 32, 0, s>>>(a, act);
  return cudaGetLastError();
}

}  // namespace rocmfp4
