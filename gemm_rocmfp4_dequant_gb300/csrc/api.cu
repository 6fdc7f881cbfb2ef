// C ABI of the ROCmFP4 library (declared in include/rocmfp4.h): host-side
// argument checks, per-device state, and kernel dispatch.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/rocmfp4.h"
#include "kernels.h"

namespace {

using namespace rocmfp4;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int occ[2][2][4] = {};             // stream kernel CTAs per SM [variant][act][log2 mb]
  int64_t wmax = 0;                  // workspace capacity in warps
  float* ws = nullptr;               // 2 * wmax records of kStreamTileRows * 8 floats
  uint32_t* cnt = nullptr;           // wmax split counters
  uint32_t* err = nullptr;           // kernel error bits
  float* tcws = nullptr;             // tensor-core kernel: split-tile partials
  uint32_t* tccnt = nullptr;         // tensor-core kernel: split-tile counters
  float* attn_ws = nullptr;          // decode attention: split partials
  unsigned long long* vfirst = nullptr;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_launches{0};
thread_local std::string t_last_error;

rocmfp4_status fail(rocmfp4_status st, const std::string& msg) {
  t_last_error = msg;
  return st;
}

rocmfp4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ROCMFP4_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_variant(int v) { return v == ROCMFP4_DUAL || v == ROCMFP4_FAST; }
bool valid_act(int a) { return a == ROCMFP4_ACT_F16 || a == ROCMFP4_ACT_BF16; }

int64_t block_bytes_of(int v) { return v == ROCMFP4_DUAL ? 18 : 17; }

// Per-device set-up on first use: SM count, kernel attributes, occupancy and
// the workspace of the split-tile reduction.
rocmfp4_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ROCMFP4_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = stream_init_driver()) != cudaSuccess) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
    if ((e = tc_prepare()) != cudaSuccess) return cuda_fail(e, "tensor-core kernel set-up");
    if ((e = attn_prepare()) != cudaSuccess) return cuda_fail(e, "attention kernel set-up");
    int best = 1;
    for (int v = 0; v < 2; ++v)
      for (int a = 0; a < 2; ++a)
        for (int lm = 0; lm < 4; ++lm) {
          int& o = d.occ[v][a][lm];
          if ((e = stream_prepare(v, a, 1 << lm)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
          if ((e = stream_occupancy(v, a, 1 << lm, &o)) != cudaSuccess) return cuda_fail(e, "occupancy");
          if (o < 1) return fail(ROCMFP4_ERR_UNSUPPORTED, "streaming kernel does not fit on this device");
          best = o > best ? o : best;
        }
    d.wmax = (int64_t)d.sms * best * kStreamWarpsPerCta;
    if ((e = cudaMalloc(&d.ws, sizeof(float) * kStreamTileRows * 8 * 2 * d.wmax)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMalloc(&d.cnt, sizeof(uint32_t) * d.wmax)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMalloc(&d.err, sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMalloc(&d.vfirst, sizeof(unsigned long long))) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemset(d.cnt, 0, sizeof(uint32_t) * d.wmax)) != cudaSuccess) return cuda_fail(e, "cudaMemset");
    if ((e = cudaMalloc(&d.tcws, sizeof(float) * tc_ws_floats(d.sms))) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMalloc(&d.tccnt, sizeof(uint32_t) * tc_cnt_words(d.sms))) != cudaSuccess)
      return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemset(d.tccnt, 0, sizeof(uint32_t) * tc_cnt_words(d.sms))) != cudaSuccess)
      return cuda_fail(e, "cudaMemset");
    if ((e = cudaMalloc(&d.attn_ws, sizeof(float) * attn_ws_floats(d.sms))) != cudaSuccess)
      return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemset(d.err, 0, sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e, "cudaMemset");
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    d.ready = true;
  }
  *out = &d;
  return ROCMFP4_OK;
}

// The state of the current device if an allocating entry point has set it
// up there, else nullptr (never creates it).
DeviceState* existing_state() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_dev[dev].ready ? &g_dev[dev] : nullptr;
}

rocmfp4_status check_shape(int64_t N, int64_t K, int variant) {
  if (!valid_variant(variant)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown variant");
  if (N < 0 || K < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative size");
  if (K % 32 != 0) return fail(ROCMFP4_ERR_INVALID_ARG, "K must be a multiple of 32");
  return ROCMFP4_OK;
}

// Warps of a single-product streaming launch for `tiles` tiles of `nspans`
// units of `unit_bytes` weight bytes, M activation rows, with room for `cap`
// warps.  Units go to warps in contiguous equal ranges, four warps to a CTA.
// When the tiles can be dealt out whole to CTAs that each stream at most
// kAlignedCtaBytes of weights (and M <= 4), the grid has one CTA per run of
// whole tiles: a tile is then split only between the warps of one CTA
// (whenever the CTAs divide the tiles evenly), and the reduction never
// takes its cross-CTA level, whose two L2 round trips at the end of the
// launch cost more than the extra warps gain.  Otherwise (long rows, or
// 8 activation rows) every warp that fits takes a share, which keeps more
// bytes in flight.
constexpr int64_t kAlignedCtaBytes = 40 * 4608;  // 40 dual units of 32 rows x 256 weights
}  // namespace

int64_t rocmfp4::stream_warps(int64_t tiles, int64_t nspans, int64_t unit_bytes, int64_t M, int64_t cap) {
  const int64_t units = tiles * nspans;
  const int64_t maxc = cap / kStreamWarpsPerCta;
  const int64_t tpc = (tiles + maxc - 1) / maxc;  // tiles per CTA
  if (M <= 4 && tpc * nspans * unit_bytes <= kAlignedCtaBytes) {
    const int64_t w = (tiles + tpc - 1) / tpc * kStreamWarpsPerCta;
    return units < w ? units : w;
  }
  return units < cap ? units : cap;
}

namespace {

rocmfp4_status product(const void* W, const void* X, float* Y, int64_t M, int64_t N, int64_t K, int variant,
                       int act, cudaStream_t s) {
  rocmfp4_status st = check_shape(N, K, variant);
  if (st != ROCMFP4_OK) return st;
  if (!valid_act(act)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown activation type");
  if (M < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative size");
  if (M == 0 || N == 0) return ROCMFP4_OK;
  if (Y == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "Y is NULL");
  if (K > 0 && W == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "W is NULL");
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(Y, 0, sizeof(float) * M * N, s);
    return e == cudaSuccess ? ROCMFP4_OK : cuda_fail(e, "cudaMemsetAsync");
  }
  if (X == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "X is NULL");
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != ROCMFP4_OK) return st;

  const int64_t row_bytes = K / 32 * block_bytes_of(variant);
  const int64_t ku = stream_weights_per_unit(variant);
  // The streaming kernel indexes units and tiles in 32 bits.
  const bool stream_ok = K % ku == 0 && aligned16(W) && aligned16(X) &&
                         (N + kStreamTileRows - 1) / kStreamTileRows * (K / ku) < (int64_t(1) << 31);
  const uint16_t* Xh = static_cast<const uint16_t*>(X);
  // More than 8 activation rows: the tensor-core kernel reads W once per
  // 256-token tile instead of once per 8 rows.
  const bool tc_ok = M > 8 && K % tc_k_multiple(variant) == 0 && aligned16(W) && aligned16(X) &&
                     M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31);
  if (tc_ok) {
    TcArgs a{static_cast<const uint8_t*>(W), Xh, Y, M, N, K, row_bytes, d->tcws, d->tccnt, d->err};
    cudaError_t e = launch_gemm_tc(variant, act, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
    g_launches.fetch_add(1);
    return ROCMFP4_OK;
  }
  if (!stream_ok || M > 8) {
    GenericArgs a{static_cast<const uint8_t*>(W), Xh, Y, N, K, row_bytes, M};
    cudaError_t e = launch_gemm_generic(variant, act, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "generic kernel launch");
    g_launches.fetch_add(1);
    return ROCMFP4_OK;
  }
  const int64_t nspans = K / ku;
  const int64_t tiles = (N + kStreamTileRows - 1) / kStreamTileRows;
  const int64_t units = tiles * nspans;
  for (int64_t m0 = 0; m0 < M; m0 += 8) {
    const int mc = (int)(M - m0 < 8 ? M - m0 : 8);
    const int mb = stream_mb_for(mc);
    const int lm = mb == 1 ? 0 : mb == 2 ? 1 : mb == 4 ? 2 : 3;
    const int64_t cap = (int64_t)d->sms * d->occ[variant][act][lm] * kStreamWarpsPerCta;
    const int64_t wact = stream_warps(tiles, nspans, ku * block_bytes_of(variant), mc, cap);
    const int ctas = (int)((wact + kStreamWarpsPerCta - 1) / kStreamWarpsPerCta);
    GemvArgs a{};
    a.W = static_cast<const uint8_t*>(W);
    a.X = Xh + m0 * K;
    a.Y = Y + m0 * N;
    a.N = N;
    a.K = K;
    a.row_bytes = row_bytes;
    a.M = mc;
    a.nspans = nspans;
    a.units = units;
    a.wact = wact;
    a.ws = d->ws;
    a.cnt = d->cnt;
    a.err = d->err;
    // A grid of at most two CTAs per SM takes the deeper rings (M <= 2).
    a.deep = mb <= 2 && ctas <= 2 * d->sms ? 1 : 0;
    cudaError_t e = launch_gemv_stream(variant, act, a, ctas, s);
    if (e != cudaSuccess) return cuda_fail(e, "streaming kernel launch");
    g_launches.fetch_add(1);
  }
  return ROCMFP4_OK;
}

rocmfp4_status chain(const rocmfp4_gemv_op* ops, int count, int64_t M, int variant, int act, cudaStream_t s) {
  if (count < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative count");
  if (count == 0) return ROCMFP4_OK;
  if (ops == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "ops is NULL");
  if (!valid_act(act)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown activation type");
  if (M < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative size");
  for (int i = 0; i < count; ++i) {
    const rocmfp4_gemv_op& op = ops[i];
    rocmfp4_status st = check_shape(op.N, op.K, variant);
    if (st != ROCMFP4_OK) return fail(st, "product " + std::to_string(i) + ": " + t_last_error);
    if (M == 0 || op.N == 0) continue;
    if (op.Y == nullptr || (op.K > 0 && (op.W == nullptr || op.X == nullptr)))
      return fail(ROCMFP4_ERR_INVALID_ARG, "product " + std::to_string(i) + ": NULL pointer");
  }
  if (M == 0) return ROCMFP4_OK;
  // One launch per product, in order, exactly as rocmfp4_gemm_ex would run
  // it.  Streaming launches are programmatic dependent launches: a product's
  // weights stream while the previous product finishes, and its activations
  // are read only once the previous launch has completed.  (One cooperative
  // launch with a grid barrier between products measured slower at every
  // size, from N = 256 to the layer's matrices.)
  for (int i = 0; i < count; ++i) {
    if (ops[i].N == 0) continue;
    rocmfp4_status st = product(ops[i].W, ops[i].X, ops[i].Y, M, ops[i].N, ops[i].K, variant, act, s);
    if (st != ROCMFP4_OK) return st;
  }
  return ROCMFP4_OK;
}

// Fused gate/up product (M <= 8): W holds 2I rows, the I gate rows then the
// I up rows; Y[m][i] = SiLU(gate_i . x_m) * (up_i . x_m).
rocmfp4_status gate_up(const void* W, const void* X, float* Y, int64_t M, int64_t I, int64_t K, int variant, int act,
                       cudaStream_t s) {
  rocmfp4_status st = check_shape(I, K, variant);
  if (st != ROCMFP4_OK) return st;
  if (!valid_act(act)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown activation type");
  if (M < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative size");
  if (M == 0 || I == 0) return ROCMFP4_OK;
  if (M > 8) return fail(ROCMFP4_ERR_UNSUPPORTED, "gate/up product: at most 8 activation rows");
  if (Y == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "Y is NULL");
  if (K > 0 && W == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "W is NULL");
  if (K == 0) {  // SiLU(0) * 0
    cudaError_t e = cudaMemsetAsync(Y, 0, sizeof(float) * M * I, s);
    return e == cudaSuccess ? ROCMFP4_OK : cuda_fail(e, "cudaMemsetAsync");
  }
  if (X == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "X is NULL");
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != ROCMFP4_OK) return st;
  const int64_t ku = stream_weights_per_unit(variant);
  const int64_t nspans = K / ku;
  const int64_t tiles = (I + kStreamTileRows / 2 - 1) / (kStreamTileRows / 2);  // 16 gate and 16 up rows each
  const int64_t units = tiles * nspans;
  if (K % ku != 0 || !aligned16(W) || !aligned16(X) || units >= (int64_t(1) << 31))
    return fail(ROCMFP4_ERR_UNSUPPORTED,
                "gate/up product: K must be a multiple of 256 (dual) or 512 (single-scale), W and X 16-byte aligned");
  const int mb = stream_mb_for((int)M);
  const int lm = mb == 1 ? 0 : mb == 2 ? 1 : mb == 4 ? 2 : 3;
  const int64_t cap = (int64_t)d->sms * d->occ[variant][act][lm] * kStreamWarpsPerCta;
  GemvArgs a{};
  a.W = static_cast<const uint8_t*>(W);
  a.X = static_cast<const uint16_t*>(X);
  a.Y = Y;
  a.N = I;
  a.K = K;
  a.row_bytes = K / 32 * block_bytes_of(variant);
  a.M = (int)M;
  a.nspans = nspans;
  a.units = units;
  a.wact = stream_warps(tiles, nspans, ku * block_bytes_of(variant), M, cap);
  a.ws = d->ws;
  a.cnt = d->cnt;
  a.err = d->err;
  a.epi = 1;
  const int ctas = (int)((a.wact + kStreamWarpsPerCta - 1) / kStreamWarpsPerCta);
  cudaError_t e = launch_gemv_stream(variant, act, a, ctas, s);
  if (e != cudaSuccess) return cuda_fail(e, "streaming kernel launch");
  g_launches.fetch_add(1);
  return ROCMFP4_OK;
}

rocmfp4_status decode_attention(const void* q, const void* K, const void* V, const int32_t* lens, float* out,
                                int64_t B, int64_t H, int64_t Hkv, int64_t D, int64_t Tmax, float scale, int variant,
                                int act, cudaStream_t s) {
  if (!valid_variant(variant)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown variant");
  if (!valid_act(act)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown activation type");
  if (B < 0 || H < 0 || Hkv < 1 || D < 0 || Tmax < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative or zero size");
  if (H % Hkv != 0) return fail(ROCMFP4_ERR_INVALID_ARG, "H must be a multiple of Hkv");
  if (D % 32 != 0) return fail(ROCMFP4_ERR_INVALID_ARG, "D must be a multiple of 32");
  if (B == 0 || H == 0) return ROCMFP4_OK;
  if (out == nullptr || q == nullptr || lens == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "NULL pointer");
  if (Tmax > 0 && (K == nullptr || V == nullptr)) return fail(ROCMFP4_ERR_INVALID_ARG, "NULL pointer");
  if (D != 64 && D != 128) return fail(ROCMFP4_ERR_UNSUPPORTED, "decode attention: D must be 64 or 128");
  if (H / Hkv > 8) return fail(ROCMFP4_ERR_UNSUPPORTED, "decode attention: at most 8 query heads per KV head");
  if (Tmax % 32 != 0) return fail(ROCMFP4_ERR_UNSUPPORTED, "decode attention: Tmax must be a multiple of 32");
  if (Tmax > 0 && (!aligned16(K) || !aligned16(V)))
    return fail(ROCMFP4_ERR_UNSUPPORTED, "decode attention: K and V must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lens) & 3u) != 0) return fail(ROCMFP4_ERR_INVALID_ARG, "lens misaligned");
  if (B * H >= (int64_t(1) << 31) || B * Hkv * Tmax >= (int64_t(1) << 40) || Tmax >= (int64_t(1) << 31))
    return fail(ROCMFP4_ERR_UNSUPPORTED, "decode attention: sizes too large");
  if (!(scale == scale)) return fail(ROCMFP4_ERR_INVALID_ARG, "scale is NaN");
  if (Tmax == 0) {  // no token anywhere: zeros
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * B * H * D, s);
    return e == cudaSuccess ? ROCMFP4_OK : cuda_fail(e, "cudaMemsetAsync");
  }
  DeviceState* d = nullptr;
  rocmfp4_status st = device_state(&d);
  if (st != ROCMFP4_OK) return st;
  AttnArgs a{static_cast<const uint16_t*>(q), static_cast<const uint8_t*>(K), static_cast<const uint8_t*>(V), lens,
             out, d->attn_ws, B, H, Hkv, D, Tmax, scale, d->err};
  int launches = 0;
  cudaError_t e = launch_decode_attention(variant, act, a, d->sms, s, &launches);
  g_launches.fetch_add((uint64_t)launches);
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  return ROCMFP4_OK;
}

}  // namespace

namespace rocmfp4 {
void set_last_error(const std::string& message) { t_last_error = message; }
void count_launch() { g_launches.fetch_add(1); }
}  // namespace rocmfp4

extern "C" {

size_t rocmfp4_block_bytes(rocmfp4_variant variant) {
  return valid_variant(variant) ? (size_t)block_bytes_of(variant) : 0;
}

size_t rocmfp4_row_bytes(int64_t K, rocmfp4_variant variant) {
  if (!valid_variant(variant) || K < 0 || K % 32 != 0) return 0;
  return (size_t)(K / 32 * block_bytes_of(variant));
}

rocmfp4_status rocmfp4_gemv(const void* W, const void* x, float* y, int64_t N, int64_t K,
                            rocmfp4_variant variant) {
  return product(W, x, y, 1, N, K, variant, ROCMFP4_ACT_F16, nullptr);
}

rocmfp4_status rocmfp4_gemv_ex(const void* W, const void* x, float* y, int64_t N, int64_t K,
                               rocmfp4_variant variant, rocmfp4_act act, rocmfp4_stream_t stream) {
  return product(W, x, y, 1, N, K, variant, act, reinterpret_cast<cudaStream_t>(stream));
}

rocmfp4_status rocmfp4_gemm(const void* W, const void* X, float* Y, int64_t M, int64_t N, int64_t K,
                            rocmfp4_variant variant) {
  return product(W, X, Y, M, N, K, variant, ROCMFP4_ACT_BF16, nullptr);
}

rocmfp4_status rocmfp4_gemm_ex(const void* W, const void* X, float* Y, int64_t M, int64_t N, int64_t K,
                               rocmfp4_variant variant, rocmfp4_act act, rocmfp4_stream_t stream) {
  return product(W, X, Y, M, N, K, variant, act, reinterpret_cast<cudaStream_t>(stream));
}

rocmfp4_status rocmfp4_gemv_gate_up(const void* W, const void* X, float* Y, int64_t M, int64_t I, int64_t K,
                                    rocmfp4_variant variant, rocmfp4_act act, rocmfp4_stream_t stream) {
  return gate_up(W, X, Y, M, I, K, variant, act, reinterpret_cast<cudaStream_t>(stream));
}

rocmfp4_status rocmfp4_decode_attention(const void* q, const void* K, const void* V, const int32_t* lens, float* out,
                                        int64_t B, int64_t H, int64_t Hkv, int64_t D, int64_t Tmax, float scale,
                                        rocmfp4_variant variant, rocmfp4_act act, rocmfp4_stream_t stream) {
  return decode_attention(q, K, V, lens, out, B, H, Hkv, D, Tmax, scale, variant, act,
                          reinterpret_cast<cudaStream_t>(stream));
}

rocmfp4_status rocmfp4_gemv_chain(const rocmfp4_gemv_op* ops, int count, int64_t M, rocmfp4_variant variant,
                                  rocmfp4_act act, rocmfp4_stream_t stream) {
  return chain(ops, count, M, variant, act, reinterpret_cast<cudaStream_t>(stream));
}

rocmfp4_status rocmfp4_gemv_chain_mixed(const rocmfp4_gemv_op* ops, const rocmfp4_variant* variants, int count,
                                        int64_t M, rocmfp4_act act, rocmfp4_stream_t stream) {
  if (count < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative count");
  if (count == 0) return ROCMFP4_OK;
  if (ops == nullptr || variants == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "ops or variants is NULL");
  if (!valid_act(act)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown activation type");
  if (M < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative size");
  // every product is checked before any launch, as in a single-layout chain
  for (int i = 0; i < count; ++i) {
    const rocmfp4_gemv_op& op = ops[i];
    rocmfp4_status st = check_shape(op.N, op.K, variants[i]);
    if (st != ROCMFP4_OK) return fail(st, "product " + std::to_string(i) + ": " + t_last_error);
    if (M == 0 || op.N == 0) continue;
    if (op.Y == nullptr || (op.K > 0 && (op.W == nullptr || op.X == nullptr)))
      return fail(ROCMFP4_ERR_INVALID_ARG, "product " + std::to_string(i) + ": NULL pointer");
  }
  // runs of products with one layout, each a single-layout chain, in order
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int i = 0; i < count;) {
    int n = 1;
    while (i + n < count && variants[i + n] == variants[i]) ++n;
    rocmfp4_status st = chain(ops + i, n, M, variants[i], act, s);
    if (st != ROCMFP4_OK) return st;
    i += n;
  }
  return ROCMFP4_OK;
}

rocmfp4_status rocmfp4_dequant(const void* W, void* out, rocmfp4_out_dtype out_dtype, int64_t N, int64_t K,
                               rocmfp4_variant variant, rocmfp4_stream_t stream) {
  rocmfp4_status st = check_shape(N, K, variant);
  if (st != ROCMFP4_OK) return st;
  if (out_dtype != ROCMFP4_OUT_F32 && out_dtype != ROCMFP4_OUT_BF16 && out_dtype != ROCMFP4_OUT_F16)
    return fail(ROCMFP4_ERR_INVALID_ARG, "unknown output type");
  const int64_t nblocks = N * (K / 32);
  if (nblocks == 0) return ROCMFP4_OK;
  if (W == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "W is NULL");
  if (out == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "out is NULL");
  cudaError_t e = launch_dequant(variant, out_dtype, static_cast<const uint8_t*>(W), out, nblocks,
                                 reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
  g_launches.fetch_add(1);
  return ROCMFP4_OK;
}

rocmfp4_status rocmfp4_quantize(const void* src, rocmfp4_act src_type, void* W, int64_t N, int64_t K,
                                rocmfp4_variant variant, rocmfp4_stream_t stream) {
  rocmfp4_status st = check_shape(N, K, variant);
  if (st != ROCMFP4_OK) return st;
  if (!valid_act(src_type)) return fail(ROCMFP4_ERR_INVALID_ARG, "unknown source type");
  const int64_t nblocks = N * (K / 32);
  if (nblocks == 0) return ROCMFP4_OK;
  if (src == nullptr || W == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "NULL pointer");
  if ((reinterpret_cast<uintptr_t>(src) & 1u) != 0) return fail(ROCMFP4_ERR_INVALID_ARG, "src misaligned");
  cudaError_t e = launch_quantize(variant, src_type, static_cast<const uint16_t*>(src), static_cast<uint8_t*>(W),
                                  nblocks, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  g_launches.fetch_add(1);
  return ROCMFP4_OK;
}

rocmfp4_status rocmfp4_copy(void* dst, const void* src, int64_t bytes, rocmfp4_stream_t stream) {
  if (bytes < 0) return fail(ROCMFP4_ERR_INVALID_ARG, "negative size");
  if (bytes == 0) return ROCMFP4_OK;
  if (dst == nullptr || src == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "NULL pointer");
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst), sp = reinterpret_cast<uintptr_t>(src);
  if ((d < sp ? sp - d : d - sp) < (uintptr_t)bytes) return fail(ROCMFP4_ERR_INVALID_ARG, "overlapping ranges");
  // Each side must be memory a kernel on the current device can address:
  // its own device memory, managed memory, or pinned host memory (through
  // its device pointer).  Pageable host memory and another device's memory
  // are refused rather than handed to the kernel.
  int cur = 0;
  cudaError_t ce = cudaGetDevice(&cur);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
  void* ends[2] = {dst, const_cast<void*>(src)};
  for (void*& p : ends) {
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
    if (at.type == cudaMemoryTypeUnregistered)
      return fail(ROCMFP4_ERR_INVALID_ARG, "pageable host memory: pin it (cudaHostAlloc / cudaHostRegister)");
    if (at.type == cudaMemoryTypeDevice && at.device != cur)
      return fail(ROCMFP4_ERR_INVALID_ARG, "device memory of another device");
    if (at.type == cudaMemoryTypeHost) {
      if (at.devicePointer == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "host memory not mapped for the device");
      p = at.devicePointer;
    }
  }
  cudaError_t e = launch_copy(ends[0], ends[1], bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy launch");
  g_launches.fetch_add(1);
  return ROCMFP4_OK;
}

rocmfp4_status rocmfp4_validate(const void* W, int64_t N, int64_t K, rocmfp4_variant variant,
                                int64_t* first_bad_block, rocmfp4_stream_t stream) {
  if (first_bad_block) *first_bad_block = -1;
  rocmfp4_status st = check_shape(N, K, variant);
  if (st != ROCMFP4_OK) return st;
  const int64_t nblocks = N * (K / 32);
  if (nblocks == 0) return ROCMFP4_OK;
  if (W == nullptr) return fail(ROCMFP4_ERR_INVALID_ARG, "W is NULL");
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != ROCMFP4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned long long first = ~0ull;
  cudaError_t e = cudaMemcpyAsync(d->vfirst, &first, sizeof(first), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  if ((e = launch_validate(variant, static_cast<const uint8_t*>(W), nblocks, d->vfirst, s)) != cudaSuccess)
    return cuda_fail(e, "validate launch");
  g_launches.fetch_add(1);
  if ((e = cudaMemcpyAsync(&first, d->vfirst, sizeof(first), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpyAsync");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (first == ~0ull) return ROCMFP4_OK;
  if (first_bad_block) *first_bad_block = (int64_t)first;
  return ROCMFP4_ERR_INVALID_SCALE;
}

uint32_t rocmfp4_device_error_bits(rocmfp4_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  // The allocating entry points' workspace, only if one exists: the query
  // itself never creates it.
  if (DeviceState* d = existing_state()) {
    if (cudaMemcpyAsync(&bits, d->err, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess) return 0xFFFFFFFFu;
    if (cudaStreamSynchronize(s) != cudaSuccess) return 0xFFFFFFFFu;
    if (bits != 0) {
      // A kernel gave up waiting: its split counters may be left set, so clear them.
      cudaMemsetAsync(d->err, 0, sizeof(uint32_t), s);
      cudaMemsetAsync(d->cnt, 0, sizeof(uint32_t) * d->wmax, s);
      cudaMemsetAsync(d->tccnt, 0, sizeof(uint32_t) * tc_cnt_words(d->sms), s);
      if (cudaStreamSynchronize(s) != cudaSuccess) return 0xFFFFFFFFu;
    }
  }
  // The allocation-free entry point's fixed array, if it was set up here.
  uint32_t nb = 0;
  if (noalloc_error_bits(s, &nb) != cudaSuccess) return 0xFFFFFFFFu;
  return bits | nb;
}

const char* rocmfp4_status_string(rocmfp4_status status) {
  switch (status) {
    case ROCMFP4_OK: return "ROCMFP4_OK";
    case ROCMFP4_ERR_INVALID_ARG: return "ROCMFP4_ERR_INVALID_ARG";
    case ROCMFP4_ERR_UNSUPPORTED: return "ROCMFP4_ERR_UNSUPPORTED";
    case ROCMFP4_ERR_INVALID_SCALE: return "ROCMFP4_ERR_INVALID_SCALE";
    case ROCMFP4_ERR_CUDA: return "ROCMFP4_ERR_CUDA";
  }
  return "ROCMFP4_UNKNOWN_STATUS";
}

const char* rocmfp4_last_error(void) { return t_last_error.c_str(); }

uint64_t rocmfp4_launch_count(void) { return g_launches.load(); }

void rocmfp4_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (int dev = 0; dev < kMaxDevices; ++dev) {
    DeviceState& d = g_dev[dev];
    if (!d.ready) continue;
    cudaSetDevice(dev);
    cudaDeviceSynchronize();
    cudaFree(d.ws);
    cudaFree(d.cnt);
    cudaFree(d.err);
    cudaFree(d.tcws);
    cudaFree(d.tccnt);
    cudaFree(d.attn_ws);
    cudaFree(d.vfirst);
    d = DeviceState{};
  }
  cudaSetDevice(cur);
}

}  // extern "C"
