// Host-side launch interface between api.cu and the kernel translation units.
#pragma once
#include <cstdint>
#include <string>
#include <cuda_runtime.h>

namespace rocmfp4 {

// Host-side bookkeeping shared by the C entry points (api.cu).
void set_last_error(const std::string& message);  // text of rocmfp4_last_error()
void count_launch();                              // one more kernel for rocmfp4_launch_count()

// Streaming product Y[M][N] = X[M][K] . W[N][K]^T for M <= 8.
struct GemvArgs {
  const uint8_t* W;      // N x row_bytes packed blocks (2N rows, gate then up, when epi)
  const uint16_t* X;     // M x K activations (fp16 or bf16 bits)
  float* Y;              // M x N outputs
  int64_t N, K, row_bytes;
  int M;
  int64_t nspans;        // K / weights-per-unit
  int64_t units;         // ceil(N/32) * nspans, or ceil(N/16) * nspans when epi
  int64_t wact;          // active warps (<= units)
  float* ws;             // 2 * wact records of 32 x 8 floats
  uint32_t* cnt;         // wact counters, zero between calls
  uint32_t* err;         // error bits
  int epi = 0;           // 1: Y = SiLU(gate rows . x) * (up rows . x)
  int deep = 0;          // 1: deeper per-warp rings, two CTAs per SM (plain products, M <= 2)
};

constexpr int kStreamWarpsPerCta = 4;
constexpr int kStreamTileRows = 32;
int stream_mb_for(int M);                   // staged activation rows: 1, 2, 4 or 8
int stream_weights_per_unit(int variant);   // 256 (dual) or 512 (single-scale)
size_t stream_smem_bytes(int variant, int mb, int deep);
cudaError_t stream_prepare(int variant, int act, int mb);  // sets the dynamic smem attribute
cudaError_t stream_occupancy(int variant, int act, int mb, int* ctas_per_sm);
cudaError_t stream_init_driver();           // resolves cuTensorMapEncodeTiled once
cudaError_t launch_gemv_stream(int variant, int act, const GemvArgs& a, int ctas, cudaStream_t s);
// Active warps of a single-product streaming launch over `tiles` tiles of
// `nspans` units of `unit_bytes` weight bytes, M activation rows, with room
// for `cap` warps (api.cu).
int64_t stream_warps(int64_t tiles, int64_t nspans, int64_t unit_bytes, int64_t M, int64_t cap);
// Error bits of the allocation-free entry point's fixed scratch on the
// current device (noalloc.cu): 0 when it has not been set up there.  Reads
// and clears them, and on a non-zero result zeroes its split counters.
cudaError_t noalloc_error_bits(cudaStream_t s, uint32_t* bits);

// Tensor-core product Y[M][N] = X[M][K] . W[N][K]^T (tcgen05, decoded weights
// in tensor memory).  Needs K % tc_k_multiple(variant) == 0, W and X 16-byte
// aligned, and M, N, K below 2^31.
struct TcArgs {
  const uint8_t* W;
  const uint16_t* X;
  float* Y;
  int64_t M, N, K, row_bytes;
  float* ws;       // split-tile partials: tc_ws_floats(sms) floats
  uint32_t* cnt;   // split-tile counters: tc_cnt_words(sms) words, zero between launches
  uint32_t* err;
};
int tc_k_multiple(int variant);   // 256 (dual) or 512 (single-scale)
size_t tc_ws_floats(int sms);     // one partial tile of 128 x 256 fp32 per SM
size_t tc_cnt_words(int sms);     // one counter per tile of the split region (at most 2 per SM)
cudaError_t tc_prepare();         // resolves cuTensorMapEncodeTiled, sets the smem attributes
cudaError_t launch_gemm_tc(int variant, int act, const TcArgs& a, cudaStream_t s);

// Decode attention over a ROCmFP4 K/V cache (attention.cu): q [B][H][D],
// K and V [B][Hkv][Tmax] rows of D/32 blocks, lens [B], out [B][H][D] fp32.
// D is 64 or 128, H / Hkv at most 8, Tmax a multiple of 32, K and V 16-byte
// aligned.  One split launch, plus a combine launch when the cache is split.
constexpr int kAttnMaxD = 128;
struct AttnArgs {
  const uint16_t* q;
  const uint8_t* K;
  const uint8_t* V;
  const int32_t* lens;
  float* out;
  float* ws;  // attn_ws_floats(sms) floats
  int64_t B, H, Hkv, D, Tmax;
  float scale;
  uint32_t* err;
};
size_t attn_ws_floats(int sms);
cudaError_t attn_prepare();
cudaError_t launch_decode_attention(int variant, int act, const AttnArgs& a, int sms, cudaStream_t s, int* launches);

// Any K % 32 == 0, any alignment: one warp per (row, column chunk).
struct GenericArgs {
  const uint8_t* W;
  const uint16_t* X;
  float* Y;
  int64_t N, K, row_bytes;
  int64_t M;
};
cudaError_t launch_gemm_generic(int variant, int act, const GenericArgs& a, cudaStream_t s);

// Dequantisation to fp32 / bf16 / fp16 (out_dtype 0/1/2), flat over blocks.
cudaError_t launch_dequant(int variant, int out_dtype, const uint8_t* W, void* out, int64_t nblocks,
                           cudaStream_t s);

// First block with a non-finite scale byte -> atomicMin into *first (init INT64_MAX).
// Quantiser fp16 / bf16 (act 0 / 1) -> ROCmFP4 blocks, one thread per block
// of 32 consecutive source values.
cudaError_t launch_quantize(int variant, int act, const uint16_t* src, uint8_t* W, int64_t nblocks, cudaStream_t s);
cudaError_t launch_validate(int variant, const uint8_t* W, int64_t nblocks, unsigned long long* first,
                            cudaStream_t s);

// Stream-ordered copy of `bytes` bytes by a kernel (programmatic dependent
// launch); each pointer is device memory or device-addressable host memory.
cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s);

}  // namespace rocmfp4
