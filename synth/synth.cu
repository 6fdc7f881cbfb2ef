// Device-side twin of synth/__init__.py: fills device buffers with the same
// seeded synthetic ROCmFP4 weight bytes and N(0,1) activations, bit for bit.
// The definition (counter-based SplitMix64, byte recipe, Box-Muller with
// series-evaluated ln/sin/cos in correctly rounded fp64) is stated in
// synth/__init__.py.  Every floating-point step uses an explicitly rounded
// intrinsic so that no multiply-add is fused and the numpy and CUDA results
// agree exactly.  This file holds no ROCmFP4 arithmetic.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed + kGamma * (stream + 1));
}

__device__ inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + kGamma * (i + 1)); }

__constant__ double kLn[14] = {
    0x1.0000000000000p+0, 0x1.5555555555555p-2, 0x1.999999999999ap-3, 0x1.2492492492492p-3,
    0x1.c71c71c71c71cp-4, 0x1.745d1745d1746p-4, 0x1.3b13b13b13b14p-4, 0x1.1111111111111p-4,
    0x1.e1e1e1e1e1e1ep-5, 0x1.af286bca1af28p-5, 0x1.8618618618618p-5, 0x1.642c8590b2164p-5,
    0x1.47ae147ae147bp-5, 0x1.2f684bda12f68p-5};
__constant__ double kSin[12] = {
    0x1.0000000000000p+0, -0x1.5555555555555p-3, 0x1.1111111111111p-7, -0x1.a01a01a01a01ap-13,
    0x1.71de3a556c734p-19, -0x1.ae64567f544e4p-26, 0x1.6124613a86d09p-33, -0x1.ae7f3e733b81fp-41,
    0x1.952c77030ad4ap-49, -0x1.2f49b46814157p-57, 0x1.71b8ef6dcf572p-66, -0x1.761b41316381ap-75};
__constant__ double kCos[12] = {
    0x1.0000000000000p+0, -0x1.0000000000000p-1, 0x1.5555555555555p-5, -0x1.6c16c16c16c17p-10,
    0x1.a01a01a01a01ap-16, -0x1.27e4fb7789f5cp-22, 0x1.1eed8eff8d898p-29, -0x1.93974a8c07c9dp-37,
    0x1.ae7f3e733b81fp-45, -0x1.6827863b97d97p-53, 0x1.e542ba4020225p-62, -0x1.0ce396db7f853p-70};
constexpr double kLn2 = 0x1.62e42fefa39efp-1;
constexpr double kHalfPi = 0x1.921fb54442d18p+0;
constexpr double kSqrtHalf = 0x1.6a09e667f3bcdp-1;

__device__ double series_ln(double u) {
  int e;
  double f = frexp(u, &e);
  if (f < kSqrtHalf) { f = __dmul_rn(f, 2.0); e -= 1; }
  double t = __ddiv_rn(__dsub_rn(f, 1.0), __dadd_rn(f, 1.0));
  double t2 = __dmul_rn(t, t);
  double s = kLn[13];
  for (int j = 12; j >= 0; --j) s = __dadd_rn(__dmul_rn(s, t2), kLn[j]);
  double lnf = __dmul_rn(__dmul_rn(t, 2.0), s);
  return __dadd_rn(__dmul_rn((double)e, kLn2), lnf);
}

__device__ void sincos_turn(double u, double* sn, double* cs) {
  double x = __dmul_rn(u, 4.0);
  double q = floor(x);
  double r = __dsub_rn(x, q);
  bool comp = r > 0.5;
  double rr = comp ? __dsub_rn(1.0, r) : r;
  double phi = __dmul_rn(rr, kHalfPi);
  double p2 = __dmul_rn(phi, phi);
  double s = kSin[11], c = kCos[11];
  for (int j = 10; j >= 0; --j) s = __dadd_rn(__dmul_rn(s, p2), kSin[j]);
  for (int j = 10; j >= 0; --j) c = __dadd_rn(__dmul_rn(c, p2), kCos[j]);
  double s0 = __dmul_rn(phi, s), c0 = c;
  double s1 = comp ? c0 : s0, c1 = comp ? s0 : c0;
  int qi = ((int)q) & 3;
  if (qi == 0) { *sn = s1; *cs = c1; }
  else if (qi == 1) { *sn = c1; *cs = -s1; }
  else if (qi == 2) { *sn = -s1; *cs = -c1; }
  else { *sn = -c1; *cs = s1; }
}

__global__ void fill_weights_kernel(uint8_t* __restrict__ W, uint64_t total, int bb, uint64_t key) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += stride) {
    uint64_t r = draw(key, g);
    uint32_t pos = (uint32_t)(g % (uint64_t)bb);
    uint8_t v;
    if (pos < 16) {
      v = (uint8_t)(r >> 56);
    } else {
      uint64_t e = 4 + (((r >> 32) * 7ull) >> 32);
      uint64_t m = (r >> 29) & 7ull;
      v = (uint8_t)((e << 3) | m);
    }
    W[g] = v;
  }
}

__global__ void fill_act_kernel(uint16_t* __restrict__ X, uint64_t count, uint64_t first, int act,
                                uint64_t key) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    uint64_t idx = first + i;
    uint64_t p = idx >> 1;
    uint64_t r1 = draw(key, 2 * p), r2 = draw(key, 2 * p + 1);
    double u1 = __dmul_rn((double)((r1 >> 11) + 1), 0x1p-53);
    double u2 = __dmul_rn((double)(r2 >> 11), 0x1p-53);
    double rho = __dsqrt_rn(__dmul_rn(series_ln(u1), -2.0));
    double sn, cs;
    sincos_turn(u2, &sn, &cs);
    double v = __dmul_rn(rho, (idx & 1) ? sn : cs);
    float f = __double2float_rn(v);
    uint16_t bits;
    if (act == 0) {
      bits = __half_as_ushort(__float2half_rn(f));
    } else {
      uint32_t b = __float_as_uint(f);
      b = b + ((b >> 16) & 1u) + 0x7FFFu;
      bits = (uint16_t)(b >> 16);
    }
    X[i] = bits;
  }
}

int grid_for(uint64_t n, int threads) {
  uint64_t g = (n + threads - 1) / threads;
  if (g > 152ull * 64) g = 152ull * 64;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

extern "C" {

// Fill W (device, N * (K/32) * B bytes, B = 18 for variant 0, 17 for variant 1).
// Returns 0, -1 on bad arguments, or a cudaError_t value.
int synth_fill_weights(void* W, int64_t N, int64_t K, int variant, uint64_t seed, uint64_t stream,
                       void* cuda_stream) {
  if (N < 0 || K < 0 || K % 32 != 0 || (variant != 0 && variant != 1)) return -1;
  int bb = variant == 0 ? 18 : 17;
  uint64_t total = (uint64_t)N * (uint64_t)(K / 32) * (uint64_t)bb;
  if (total == 0) return 0;
  if (!W) return -1;
  fill_weights_kernel<<<grid_for(total, 256), 256, 0, (cudaStream_t)cuda_stream>>>(
      (uint8_t*)W, total, bb, stream_key(seed, stream));
  return (int)cudaGetLastError();
}

// Fill X (device, count uint16 bit patterns) with activation elements
// first .. first+count-1 of a stream; act 0 = fp16, 1 = bf16.
int synth_fill_act(void* X, int64_t count, int64_t first, int act, uint64_t seed, uint64_t stream,
                   void* cuda_stream) {
  if (count < 0 || first < 0 || (act != 0 && act != 1)) return -1;
  if (count == 0) return 0;
  if (!X) return -1;
  fill_act_kernel<<<grid_for((uint64_t)count, 128), 128, 0, (cudaStream_t)cuda_stream>>>(
      (uint16_t*)X, (uint64_t)count, (uint64_t)first, act, stream_key(seed, stream));
  return (int)cudaGetLastError();
}

}  // extern "C"
