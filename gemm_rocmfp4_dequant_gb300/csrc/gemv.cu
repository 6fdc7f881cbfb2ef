// Streaming ROCmFP4 GEMV / small-batch product on sm_103a.
//
//   Y[m][n] = sum_k w[n][k] * X[m][k],  m < M <= 8,  fp32 accumulation.
//
// Decode path: "Feasibility Report: Porting ROCmFP4 to Atlas", section "What
// is ROCmFP4?" (Block Layout, Codebook10 Value Table, Scale Format); common.cuh
// explains how the Blackwell e2m1/e4m3 conversions reproduce it exactly.
//
// Work decomposition (stream-K over warps).  The matrix is cut into units of
// 16 rows x SPAN bytes (8 dual blocks = 144 B, or 16 single-scale blocks =
// 272 B, per row).  Units are ordered tile-major (all K spans of rows 0..15,
// then rows 16..31, ...) and every active warp of a persistent grid takes an
// equal contiguous range of them, so every warp streams the same number of
// bytes.  A warp streams its units through a private ring of shared-memory
// stages filled by 1-D bulk copies (one per row, lanes 0..15), one mbarrier
// per stage.
//
// Per unit, lane (q = lane/4, c = lane%4) owns rows q and q+8 and the
// 4-byte-aligned lane span c (BPL whole blocks) of each row.  Each block is
// eight mma.m16n8k16 steps: step s feeds qs bytes 2s and 2s+1 of the lane's
// block; each byte becomes one f16x2 A register (low nibble -> weight 2s or
// 2s+1 of half 0, high nibble -> the weight 16 further on, in half 1),
// already multiplied by the half-scale pair.  B column n holds activation
// vector n (zero for n >= M), permuted the same way.  D is flushed into
// round-to-nearest fp32 registers after every block (8 MMAs), so the tensor
// core's own accumulation never runs long.
//
// A tile (16 rows) whose units are split between warps is finished by its
// last-arriving warp: each contributor writes its 16 x 8 partial to the
// workspace, fences, and bumps a per-tile counter; the warp that completes
// the count sums all partials in warp (= K) order, writes Y and resets the
// counter.  Nobody waits and the sum order is fixed, so results are bitwise
// reproducible.
#include "common.cuh"
#include "kernels.h"

namespace rocmfp4 {
namespace {

constexpr int kWarps = kStreamWarpsPerCta;

template <int V>
constexpr int stages() { return V == 0 ? 6 : 4; }

template <int V>
constexpr int stage_bytes() { return 16 * Fmt<V>::SPAN; }

template <int V>
constexpr size_t smem_bytes() {
  return (size_t)kWarps * stages<V>() * stage_bytes<V>() + (size_t)kWarps * stages<V>() * 8;
}

__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t U, int64_t wact) {
  return ((u + 1) * wact - 1) / U;
}

// E2M1 pair of the byte at (unrolled, hence constant) position pos of a word array.
template <int SW>
RF4_DEV uint32_t e2m1x2_at(const uint32_t (&w)[SW], int pos) {
  const uint32_t word = w[pos >> 2];
  switch (pos & 3) {
    case 0: return e2m1x2<0>(word);
    case 1: return e2m1x2<1>(word);
    case 2: return e2m1x2<2>(word);
    default: return e2m1x2<3>(word);
  }
}

// Scale pair of block phi of a lane span (f16x2 of the E4M3 values).
template <int V, int SW>
RF4_DEV uint32_t scale_pair_at(const uint32_t (&w)[SW], int phi) {
  const int P = phi * Fmt<V>::BB + 16;
  if constexpr (V == 0) {
    return (P & 2) ? e4m3x2<1>(w[P >> 2]) : e4m3x2<0>(w[P >> 2]);
  } else {
    const uint32_t dup = __byte_perm(w[P >> 2], 0u, (uint32_t)(P & 3) * 0x11u);
    return e4m3x2<0>(dup);
  }
}

template <int ACT>
RF4_DEV uint32_t weight_pair(uint32_t codes_f16x2, uint32_t s2) {
  const uint32_t w = hmul2(clamp5(codes_f16x2), s2);
  if constexpr (ACT == 1) return f16x2_to_bf16x2(w);
  return w;
}

template <int V, int ACT>
__global__ void __launch_bounds__(kWarps * 32) gemv_stream_kernel(const GemvArgs p) {
  using F = Fmt<V>;
  constexpr int NS = stages<V>();
  constexpr int SW = F::SW;
  extern __shared__ __align__(128) uint8_t smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t wg = (int64_t)blockIdx.x * kWarps + warp;
  if (wg >= p.wact) return;

  uint8_t* ring = smem + (size_t)warp * NS * stage_bytes<V>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * NS * stage_bytes<V>()) + warp * NS;

  const int64_t U = p.units, S = p.nspans;
  const int64_t u0 = U * wg / p.wact, u1 = U * (wg + 1) / p.wact;
  const int64_t nunits = u1 - u0;
  const int64_t t_first = u0 / S;

  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int64_t u, int st) {
    const int64_t t = u / S, j = u % S;
    const int64_t row0 = t * 16;
    const int nvalid = (int)(p.N - row0 < 16 ? p.N - row0 : 16);
    const uint32_t bar = smem_addr(&bars[st]);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nvalid * F::SPAN));
    __syncwarp();
    if (lane < nvalid) {
      const uint8_t* src = p.W + (row0 + lane) * p.row_bytes + j * F::SPAN;
      bulk_g2s(smem_addr(ring + (size_t)st * stage_bytes<V>() + lane * F::SPAN), src, F::SPAN, bar);
    }
  };

  const int q = lane >> 2, c = lane & 3;
  const bool bcol = q < p.M;  // this lane holds B column q
  const uint16_t* xrow = p.X + (int64_t)(bcol ? q : 0) * p.K;

  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  // Writes this warp's sums for tile t (spans [js, je)), finishing the tile
  // if this warp is its last contributor.
  auto finish_tile = [&](int64_t t, int64_t js, int64_t je) {
    const int64_t ra = t * 16 + q, rb = ra + 8;
    const int c0 = 2 * c, c1 = 2 * c + 1;
    float v[4] = {acc[0], acc[1], acc[2], acc[3]};
    bool store = true;
    if (!(js == 0 && je == S)) {
      const int slot = (t == t_first) ? 0 : 1;
      float* rec = p.ws + (2 * wg + slot) * 128;
      rec[q * 8 + c0] = v[0];
      rec[q * 8 + c1] = v[1];
      rec[(q + 8) * 8 + c0] = v[2];
      rec[(q + 8) * 8 + c1] = v[3];
      __threadfence();
      __syncwarp();
      const int64_t wf = owner_of(t * S, U, p.wact), wl = owner_of(t * S + S - 1, U, p.wact);
      uint32_t old = 0;
      if (lane == 0) old = atomicAdd(&p.cnt[wf], 1u);
      old = __shfl_sync(0xffffffffu, old, 0);
      store = (int64_t)old == wl - wf;
      if (store) {
        __threadfence();
        v[0] = v[1] = v[2] = v[3] = 0.f;
        for (int64_t w2 = wf; w2 <= wl; ++w2) {
          const int64_t tf2 = (U * w2 / p.wact) / S;
          const float* r2 = p.ws + (2 * w2 + (t == tf2 ? 0 : 1)) * 128;
          v[0] += __ldcg(r2 + q * 8 + c0);
          v[1] += __ldcg(r2 + q * 8 + c1);
          v[2] += __ldcg(r2 + (q + 8) * 8 + c0);
          v[3] += __ldcg(r2 + (q + 8) * 8 + c1);
        }
        if (lane == 0) atomicExch(&p.cnt[wf], 0u);
      }
    }
    if (store) {
      if (c0 < p.M) {
        if (ra < p.N) p.Y[c0 * p.N + ra] = v[0];
        if (rb < p.N) p.Y[c0 * p.N + rb] = v[2];
      }
      if (c1 < p.M) {
        if (ra < p.N) p.Y[c1 * p.N + ra] = v[1];
        if (rb < p.N) p.Y[c1 * p.N + rb] = v[3];
      }
    }
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
  };

  for (int i = 0; i < NS - 1 && i < nunits; ++i) issue(u0 + i, i);

  int64_t js = u0 % S;  // first span of the current tile segment
  bool failed = false;
  int64_t i = 0;
  for (; i < nunits; ++i) {
    const int64_t u = u0 + i;
    const int st = (int)(i % NS);
    if (i + NS - 1 < nunits) issue(u + NS - 1, (int)((i + NS - 1) % NS));
    if (!mbar_wait_bounded(smem_addr(&bars[st]), (uint32_t)((i / NS) & 1))) {
      failed = true;
      break;
    }
    const int64_t t = u / S, j = u % S;

    const uint8_t* sbase = ring + (size_t)st * stage_bytes<V>() + c * F::LANE_BYTES;
    uint32_t wa[SW], wb[SW];
#pragma unroll
    for (int k = 0; k < SW; ++k) {
      wa[k] = reinterpret_cast<const uint32_t*>(sbase + q * F::SPAN)[k];
      wb[k] = reinterpret_cast<const uint32_t*>(sbase + (q + 8) * F::SPAN)[k];
    }

#pragma unroll
    for (int phi = 0; phi < F::BPL; ++phi) {
      const uint32_t s2a = scale_pair_at<V>(wa, phi);
      const uint32_t s2b = scale_pair_at<V>(wb, phi);
      const int64_t blk = j * (4 * F::BPL) + c * F::BPL + phi;
      uint32_t xv[16];
      if (bcol) {
        const uint4* xs = reinterpret_cast<const uint4*>(xrow + blk * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = __ldg(xs + k);
          xv[4 * k] = v.x;
          xv[4 * k + 1] = v.y;
          xv[4 * k + 2] = v.z;
          xv[4 * k + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) xv[k] = 0u;
      }
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int pos = phi * F::BB + 2 * s;
        uint32_t a[4];
        a[0] = weight_pair<ACT>(e2m1x2_at(wa, pos), s2a);
        a[1] = weight_pair<ACT>(e2m1x2_at(wb, pos), s2b);
        a[2] = weight_pair<ACT>(e2m1x2_at(wa, pos + 1), s2a);
        a[3] = weight_pair<ACT>(e2m1x2_at(wb, pos + 1), s2b);
        // B rows (2c, 2c+1) = (x[2s], x[2s+16]); rows (2c+8, 2c+9) = (x[2s+1], x[2s+17]).
        const uint32_t b0 = __byte_perm(xv[s], xv[8 + s], 0x5410);
        const uint32_t b1 = __byte_perm(xv[s], xv[8 + s], 0x7632);
        mma16816(d, a, b0, b1, ACT == 1);
      }
      acc[0] += d[0];
      acc[1] += d[1];
      acc[2] += d[2];
      acc[3] += d[3];
    }
    __syncwarp();
    fence_proxy_async();

    const bool tile_end = (j == S - 1) || (i == nunits - 1);
    if (tile_end) {
      finish_tile(t, js, j + 1);
      js = 0;
    }
  }

  if (failed) {
    if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
    // Let every copy already issued land before the shared memory is released.
    for (int64_t k = i; k < nunits && k < i + NS; ++k)
      (void)mbar_wait_bounded(smem_addr(&bars[k % NS]), (uint32_t)((k / NS) & 1));
  }
}

template <int V, int ACT>
const void* stream_kernel_ptr() {
  return reinterpret_cast<const void*>(&gemv_stream_kernel<V, ACT>);
}

const void* stream_kernel(int variant, int act) {
  if (variant == 0) return act == 0 ? stream_kernel_ptr<0, 0>() : stream_kernel_ptr<0, 1>();
  return act == 0 ? stream_kernel_ptr<1, 0>() : stream_kernel_ptr<1, 1>();
}

}  // namespace

int stream_weights_per_unit(int variant) { return variant == 0 ? Fmt<0>::KU : Fmt<1>::KU; }

size_t stream_smem_bytes(int variant) { return variant == 0 ? smem_bytes<0>() : smem_bytes<1>(); }

cudaError_t stream_prepare(int variant, int act) {
  return cudaFuncSetAttribute(stream_kernel(variant, act), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)stream_smem_bytes(variant));
}

cudaError_t stream_occupancy(int variant, int act, int* ctas_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, stream_kernel(variant, act), kWarps * 32,
                                                       stream_smem_bytes(variant));
}

cudaError_t launch_gemv_stream(int variant, int act, const GemvArgs& a, int ctas, cudaStream_t s) {
  const size_t smem = stream_smem_bytes(variant);
  if (variant == 0) {
    if (act == 0) gemv_stream_kernel<0, 0><<<ctas, kWarps * 32, smem, s>>>(a);
    else gemv_stream_kernel<0, 1><<<ctas, kWarps * 32, smem, s>>>(a);
  } else {
    if (act == 0) gemv_stream_kernel<1, 0><<<ctas, kWarps * 32, smem, s>>>(a);
    else gemv_stream_kernel<1, 1><<<ctas, kWarps * 32, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace rocmfp4
