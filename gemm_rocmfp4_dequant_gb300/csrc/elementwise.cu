// Elementwise ROCmFP4 kernels: dequantisation, scale validation, the
// quantiser (fp16 / bf16 -> ROCmFP4 blocks), the generic product used
// when a shape or pointer alignment does not fit the streaming kernel, and
// the staging copy that moves a decode step's inputs and outputs between
// pinned host memory and the device inside a chain of dependent launches.
// Decode follows "Feasibility Report: Porting ROCmFP4 to Atlas", section
// "What is ROCmFP4?" (Block Layout, Codebook10 Value Table, Scale Format), in
// plain fp32 arithmetic that is exact for every weight; the quantiser inverts
// it with the smallest covering scale and nearest codes, by exact comparisons.
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

// ---- quantiser: fp16 / bf16 -> ROCmFP4, one thread per block --------------------
// Scale groups are the two 16-weight halves (dual) or the whole block
// (single-scale).  A group's scale byte is the smallest e <= 0x7E whose
// half-scale covers its largest magnitude, 5 * E4M3(e) >= amax (0x7E when
// none does; 0 for a group of zeros); each weight takes the nearest
// Codebook10 magnitude, ties to the smaller, by comparing |x| with the
// midpoints times the half-scale.  Every product and comparison is exact in
// fp32.  Non-finite inputs count as 0.

// E4M3 value of a scale byte (bit 7 clear), exact.
RF4_DEV float ue4m3_f32(uint32_t e) {
  const uint32_t E = (e >> 3) & 15u, M = e & 7u;
  return E ? __uint_as_float(((E + 120u) << 23) | (M << 20)) : (float)M * (1.0f / 512.0f);
}

// The scale byte of a group: E4M3 values increase with the byte, so this is
// the smallest e with 5 * E4M3(e) >= amax.  A candidate comes from the fp32
// bits of amax * 0.2 (E4M3 rounded up: within one step of the answer, as the
// estimate is within a few ulp of amax / 5); one exact check each way (5 *
// E4M3(e) is exact in fp32) then fixes it.
RF4_DEV uint32_t quant_scale(float amax) {
  if (!(amax > 0.f)) return 0u;
  if (5.f * ue4m3_f32(0x7Eu) < amax) return 0x7Eu;
  const float t = amax * 0.2f;
  uint32_t e;
  if (t >= 0.015625f) {  // 2^-6 and up: E4M3 exponent field E >= 1
    const uint32_t b = __float_as_uint(t);
    uint32_t E = (b >> 23) - 120u, M = (b >> 20) & 7u;
    if (b & 0xFFFFFu) ++M;  // round the 3-bit mantissa up
    if (M == 8u) {
      M = 0u;
      ++E;
    }
    e = E > 15u ? 0x7Eu : (E << 3) | M;
  } else {  // subnormal E4M3: value M / 512
    e = (uint32_t)ceilf(t * 512.f);  // at most 8, which is 2^-6 (E = 1, M = 0)
  }
  e = e > 0x7Eu ? 0x7Eu : (e == 0u ? 1u : e);
  if (e > 1u && 5.f * ue4m3_f32(e - 1u) >= amax) --e;
  else if (5.f * ue4m3_f32(e) < amax) ++e;
  return e;
}

// The Codebook10 midpoints 0.5, 1.5, 2.5, 3.5, 5, 7, 9 as fp16 (ACT = 0) or
// bf16 bits, in both lanes.
template <int ACT>
RF4_HOSTDEV constexpr uint32_t mid_pair(int j) {
  constexpr uint32_t f16[7] = {0x3800u, 0x3E00u, 0x4100u, 0x4300u, 0x4500u, 0x4700u, 0x4880u};
  constexpr uint32_t bf16[7] = {0x3F00u, 0x3FC0u, 0x4020u, 0x4060u, 0x40A0u, 0x40E0u, 0x4110u};
  return ACT == 0 ? f16[j] | (f16[j] << 16) : bf16[j] | (bf16[j] << 16);
}

// Packed source pairs.  Every threshold of the rule, a Codebook10 midpoint
// (0.5, 1.5, 2.5, 3.5, 5, 7, 9) times a half-scale (at most 4 significant
// bits, 2^-10 .. 224), has at most 8 significant bits and lies in
// [2^-11, 2016]: it is exact in fp16 and in bf16, so comparing a source value
// with it in the source's own 16-bit format is the exact comparison.  Two
// values are compared per instruction, and the thresholds themselves are
// packed products (exact).
template <int ACT>
struct Pack {
  // |x| per lane with non-finite lanes set to 0 (they count as 0)
  static RF4_DEV uint32_t clean_abs(uint32_t w) {
    const uint32_t a = w & 0x7FFF7FFFu;
    uint32_t fin;  // 0xFFFF per lane with a <= the largest finite value
    if constexpr (ACT == 0)
      asm("set.le.u32.f16x2 %0, %1, %2;" : "=r"(fin) : "r"(a), "r"(0x7BFF7BFFu));
    else
      asm("set.le.u32.bf16x2 %0, %1, %2;" : "=r"(fin) : "r"(a), "r"(0x7F7F7F7Fu));
    return a & fin;
  }
  // the exactly representable f in both lanes
  static RF4_DEV uint32_t broadcast(float f) {
    uint32_t h;
    if constexpr (ACT == 0)
      asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(h) : "f"(f));
    else
      asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(h) : "f"(f));
    return h;
  }
  // the thresholds mid[j] * hs of a half-scale pair hs2 (exact products)
  static RF4_DEV void thresholds(uint32_t hs2, uint32_t (&t)[7]) {
#pragma unroll
    for (int j = 0; j < 7; ++j) {
      if constexpr (ACT == 0)
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t[j]) : "r"(hs2), "r"(mid_pair<ACT>(j)));
      else
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(t[j]) : "r"(hs2), "r"(mid_pair<ACT>(j)));
    }
  }
  // per lane: 0xFFFF if a > t, else 0
  static RF4_DEV uint32_t gt_mask(uint32_t a, uint32_t t) {
    uint32_t g;
    if constexpr (ACT == 0)
      asm("set.gt.u32.f16x2 %0, %1, %2;" : "=r"(g) : "r"(a), "r"(t));
    else
      asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(g) : "r"(a), "r"(t));
    return g;
  }
  static RF4_DEV float to_f32(uint32_t h) {
    if constexpr (ACT == 0)
      return __half2float(__ushort_as_half((uint16_t)h));
    else
      return __uint_as_float(h << 16);
  }
};

// Codes of the pair w (same scale group) for the thresholds t[0..6] of its
// half-scale: the nearest Codebook10 magnitude, ties to the smaller, sign in
// bit 3, zero (and any value that counts as 0) code 0.  Low lane in bits 0-3,
// high lane in bits 16-19.
template <int ACT>
RF4_DEV uint32_t pair_codes(uint32_t w, uint32_t a, const uint32_t (&t)[7]) {
  // k = #{j : a > t[j]} per lane by binary search over the increasing
  // thresholds: a > t[3] iff k >= 4, then t[5] or t[1], then one of t[6],
  // t[4], t[2], t[0]; the per-lane masks select the next threshold.
  const uint32_t g1 = Pack<ACT>::gt_mask(a, t[3]);
  const uint32_t g2 = Pack<ACT>::gt_mask(a, (g1 & t[5]) | (~g1 & t[1]));
  const uint32_t hi = (g1 & t[6]) | (~g1 & t[2]), lo = (g1 & t[4]) | (~g1 & t[0]);
  const uint32_t g3 = Pack<ACT>::gt_mask(a, (g2 & hi) | (~g2 & lo));
  const uint32_t k = (g1 & 0x00040004u) | (g2 & 0x00020002u) | (g3 & 0x00010001u);
  // sign bit 15 / 31 to bit 3 / 19 of the lanes with a nonzero count
  const uint32_t nz = (k + 0x00070007u) & 0x00080008u;  // bit 3 of a lane set iff its k != 0
  return k | ((w >> 12) & nz);
}

constexpr int kQuantThreads = 128;

template <int V, int ACT>
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const uint16_t* __restrict__ src,
                                                                   uint8_t* __restrict__ W, int64_t nblocks, bool vec,
                                                                   bool wvec) {
  using F = Fmt<V>;
  // Per warp: its 32 source blocks staged by coalesced 16-byte loads (64
  // bytes each, 16 bytes of padding after each so the per-block reads hit
  // distinct banks), and its 32 output blocks (contiguous, 18 or 17 bytes
  // each) staged for coalesced 16-byte stores.
  __shared__ __align__(16) uint8_t in_stage[kQuantThreads / 32][32 * 80];
  __shared__ __align__(16) uint8_t out_stage[kQuantThreads / 32][32 * 18];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk - lane < nblocks;
       blk += (int64_t)gridDim.x * blockDim.x) {
    // the warp's 32 blocks are all in range (a warp-uniform test)
    const bool full = blk - lane + 32 <= nblocks;
    uint32_t w[16];  // w[i] = (value 2i, value 2i+1)
    const uint16_t* s = src + blk * 32;
    if (vec && full) {
      const uint4* g = reinterpret_cast<const uint4*>(src + (blk - lane) * 32);
      __syncwarp();  // the previous step's reads of the stage are done
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ci = q * 32 + lane;  // chunk ci of the warp's 2 KB: block ci / 4, part ci % 4
        *reinterpret_cast<uint4*>(&in_stage[wib][(ci >> 2) * 80 + (ci & 3) * 16]) = g[ci];
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(&in_stage[wib][lane * 80 + q * 16]);
        w[4 * q] = v.x;
        w[4 * q + 1] = v.y;
        w[4 * q + 2] = v.z;
        w[4 * q + 3] = v.w;
      }
    } else if (blk >= nblocks) {
      continue;  // a lane past the end of a partial warp
    } else if (vec) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = reinterpret_cast<const uint4*>(s)[q];
        w[4 * q] = v.x;
        w[4 * q + 1] = v.y;
        w[4 * q + 2] = v.z;
        w[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = (uint32_t)s[2 * i] | ((uint32_t)s[2 * i + 1] << 16);
    }
    // value i: w[i / 2] half i % 2; scale group 0 = values 0..15, group 1 = 16..31 (dual)
    uint32_t a[16];
    uint32_t m0 = 0, m1 = 0;  // largest |value| bits per group and lane: non-negative values order as their bits
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      a[i] = Pack<ACT>::clean_abs(w[i]);
      if (i < 8) m0 = __vmaxu2(m0, a[i]);
      else m1 = __vmaxu2(m1, a[i]);
    }
    const float am0 = Pack<ACT>::to_f32(max(m0 & 0xFFFFu, m0 >> 16)), am1 = Pack<ACT>::to_f32(max(m1 & 0xFFFFu, m1 >> 16));
    uint32_t e0, e1;
    if constexpr (V == 0) {
      e0 = quant_scale(am0);
      e1 = quant_scale(am1);
    } else {
      e0 = e1 = quant_scale(fmaxf(am0, am1));
    }
    const float hs0 = 0.5f * ue4m3_f32(e0), hs1 = 0.5f * ue4m3_f32(e1);
    // thresholds: midpoints of the magnitudes {0,1,2,3,4,6,8,10} times the half-scale
    // (a zero half-scale gives zero thresholds, and a group of zeros gives codes 0)
    uint32_t t0[7], t1[7];
    Pack<ACT>::thresholds(Pack<ACT>::broadcast(hs0), t0);
    Pack<ACT>::thresholds(Pack<ACT>::broadcast(hs1), t1);
    // byte j: value j (low nibble, group 0) and value j + 16 (high nibble, group 1);
    // o16[i] = bytes 2i and 2i+1 = codes of values 2i, 2i+16, 2i+1, 2i+17
    uint32_t o16[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t cl = pair_codes<ACT>(w[i], a[i], t0), ch = pair_codes<ACT>(w[8 + i], a[8 + i], t1);
      o16[i] = (cl & 0xFu) | ((ch & 0xFu) << 4) | ((cl >> 16) << 8) | ((ch >> 16) << 12);
    }
    const bool coop = wvec && full;  // the warp's output (32 blocks, a multiple of 16 bytes) is 16-byte aligned
    uint8_t* out = coop ? &out_stage[wib][lane * F::BB] : W + blk * F::BB;
    if (coop) __syncwarp();  // the previous step's reads of the output stage are done
    if constexpr (V == 0) {  // 18-byte blocks start on even addresses: nine 16-bit stores
      uint16_t* p16 = reinterpret_cast<uint16_t*>(out);
#pragma unroll
      for (int k = 0; k < 8; ++k) p16[k] = (uint16_t)o16[k];
      p16[8] = (uint16_t)(e0 | (e1 << 8));
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        out[2 * k] = (uint8_t)o16[k];
        out[2 * k + 1] = (uint8_t)(o16[k] >> 8);
      }
      out[16] = (uint8_t)e0;
    }
    if (coop) {
      __syncwarp();
      constexpr int kChunks = 32 * F::BB / 16;  // 36 or 34
      uint4* g = reinterpret_cast<uint4*>(W + (blk - lane) * F::BB);
      const uint4* st = reinterpret_cast<const uint4*>(out_stage[wib]);
      g[lane] = st[lane];
      if (lane < kChunks - 32) g[32 + lane] = st[32 + lane];
    }
  }
}

// ---- staging copy (host <-> device, either side pinned host or device) -------------
// Launched with programmatic dependent launch: the next kernel on the stream
// may begin launching at once (a following product's weights then stream
// while this copy runs), and nothing is read or written before the preceding
// kernel has completed.  One 16-byte vector per thread when both pointers are
// 16-byte aligned (the tail and unaligned copies go byte by byte).
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint8_t* __restrict__ dst,
                                                             const uint8_t* __restrict__ src, int64_t bytes,
                                                             bool vec) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int64_t tid = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * kCopyThreads;
  int64_t done = 0;
  if (vec) {
    const int64_t n16 = bytes >> 4;
    for (int64_t i = tid; i < n16; i += nth) reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
    done = n16 << 4;
  }
  for (int64_t i = done + tid; i < bytes; i += nth) dst[i] = src[i];
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

cudaError_t launch_quantize(int variant, int act, const uint16_t* src, uint8_t* W, int64_t nblocks, cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const bool wvec = (reinterpret_cast<uintptr_t>(W) & 15u) == 0;
  const int threads = kQuantThreads, grid = grid_for(nblocks, threads);
  if (variant == 0) {
    if (act == 0) quantize_kernel<0, 0><<<grid, threads, 0, s>>>(src, W, nblocks, vec, wvec);
    else quantize_kernel<0, 1><<<grid, threads, 0, s>>>(src, W, nblocks, vec, wvec);
  } else {
    if (act == 0) quantize_kernel<1, 0><<<grid, threads, 0, s>>>(src, W, nblocks, vec, wvec);
    else quantize_kernel<1, 1><<<grid, threads, 0, s>>>(src, W, nblocks, vec, wvec);
  }
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

cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s) {
  if (bytes <= 0) return cudaSuccess;
  const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_for(vec ? (bytes + 15) / 16 : bytes, kCopyThreads));
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_kernel, static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), bytes,
                            vec);
}

}  // namespace rocmfp4
