// Device helpers shared by the ROCmFP4 kernels (sm_103a).
//
// Block format ("Feasibility Report: Porting ROCmFP4 to Atlas", section
// "What is ROCmFP4?", subsections "Block Layout", "Codebook10 Value Table",
// "Scale Format"): qs[16] packed 4-bit codes (byte j: weight j in the low
// nibble, weight j+16 in the high nibble), then one or two unsigned-E4M3
// scale bytes; weight = Codebook10[q] * E4M3(e) / 2.
//
// The hot decode uses the Blackwell conversion cvt.rn.f16x2.e2m1x2: a code q
// read as OCP E2M1 is exactly Codebook10[q] / 2 for every q except the two
// magnitude-7 codes (E2M1 6.0 where Codebook10 / 2 is 5.0), so a signed clamp
// of the magnitude to 5 (min.xorsign.abs) gives Codebook10[q] / 2 for all 16
// codes.  Multiplying by the E4M3 value of the scale (cvt.rn.f16x2.e4m3x2)
// then gives Codebook10[q] * hs exactly: the product has at most 7
// significant bits and lies in [2^-10, 2240], inside fp16's exact range.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#define RF4_DEV __device__ __forceinline__
#define RF4_HOSTDEV __host__ __device__ __forceinline__

namespace rocmfp4 {

// Error bits a kernel may record in the workspace error word.
enum : uint32_t { kErrWaitTimeout = 1u };

template <int V>
struct Fmt {
  static constexpr int BB = V == 0 ? 18 : 17;           // bytes per block
  static constexpr int BPL = V == 0 ? 2 : 4;            // blocks per lane per unit
  static constexpr int LANE_BYTES = BPL * BB;           // 36 / 68 (multiple of 4)
  static constexpr int SW = LANE_BYTES / 4;             // words per lane per row
  static constexpr int SPAN = 4 * LANE_BYTES;           // bytes per row per unit: 144 / 272 (multiple of 16)
  static constexpr int KU = 4 * BPL * 32;               // weights per row per unit: 256 / 512
  static constexpr int NSCALE = V == 0 ? 2 : 1;
};

RF4_DEV uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---- mbarrier + bulk copy (async proxy) ------------------------------------
RF4_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
RF4_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
RF4_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

RF4_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
RF4_DEV void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled tensor copy global -> shared (box of the tensor map at element
// coordinates (x, y)), completing the box's bytes on `bar`.
RF4_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 3-D tiled tensor copy global -> shared (box at element coordinates
// (x, y, z)), completing the box's bytes on `bar`.
RF4_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// 2-D tiled tensor copy shared -> global of the box at (x, y); elements
// outside the tensor are not written.  Part of the thread's bulk group.
RF4_DEV void tma_store_2d(const CUtensorMap* map, int32_t x, int32_t y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
RF4_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read their source.
template <int N>
RF4_DEV void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's bulk groups have completed.
RF4_DEV void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

RF4_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after about 2^32 SM cycles (seconds), returning false.
RF4_DEV bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1ll << 32)) return false;
  }
  return true;
}

// ---- programmatic dependent launch -------------------------------------------
// Wait until the grids this one depends on have completed and their writes
// are visible (a no-op when the launch has no programmatic dependency).
RF4_DEV void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid on the stream to begin launching.
RF4_DEV void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- inter-warp hand-off (split tiles) ----------------------------------------
// Release orders this thread's earlier stores (and, through __syncwarp, its
// warp's) before the increment; acquire orders later loads after it.
RF4_DEV uint32_t atomic_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
RF4_DEV void store_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- decode ------------------------------------------------------------------
// Two E2M1 codes (byte B of w: low nibble -> low half) to f16x2.
template <int B>
RF4_DEV uint32_t e2m1x2(uint32_t w) {
  uint32_t h;
  if constexpr (B == 0)
    asm("{\n .reg .b8 b;\n mov.b32 {b, _, _, _}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(h) : "r"(w));
  else if constexpr (B == 1)
    asm("{\n .reg .b8 b;\n mov.b32 {_, b, _, _}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(h) : "r"(w));
  else if constexpr (B == 2)
    asm("{\n .reg .b8 b;\n mov.b32 {_, _, b, _}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(h) : "r"(w));
  else
    asm("{\n .reg .b8 b;\n mov.b32 {_, _, _, b}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(h) : "r"(w));
  return h;
}

// Two E4M3 bytes (half H of w: byte 2H -> low half, 2H+1 -> high half) to f16x2.
template <int H>
RF4_DEV uint32_t e4m3x2(uint32_t w) {
  uint32_t h;
  if constexpr (H == 0)
    asm("{\n .reg .b16 t;\n mov.b32 {t, _}, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(h) : "r"(w));
  else
    asm("{\n .reg .b16 t;\n mov.b32 {_, t}, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(h) : "r"(w));
  return h;
}

// sign(h) * min(|h|, 5) per half: maps E2M1 +-6 to +-5 and keeps the rest.
RF4_DEV uint32_t clamp5(uint32_t h) {
  uint32_t r;
  asm("min.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x45004500u));
  return r;
}

RF4_DEV uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Exact f16x2 -> bf16x2 for values that bf16 represents exactly.
RF4_DEV uint32_t f16x2_to_bf16x2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  float lo = __low2float(v), hi = __high2float(v);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

RF4_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, bool bf16) {
  if (bf16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B into a fresh accumulator (C is zero).
RF4_DEV void mma16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, bool bf16) {
  const float z = 0.f;
  if (bf16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

// ---- scalar decode used by the dequant / validate / generic kernels ------------
// Half-scale of a (finite) scale byte as an exact fp32: E4M3(e) / 2.
RF4_DEV float halfscale_f32(uint32_t e) {
  const uint32_t E = (e >> 3) & 0xFu, M = e & 7u;
  if (E == 0) return (float)M * 0x1p-10f;                      // (M/8) * 2^-6 / 2
  return __uint_as_float(((e & 0x7Fu) << 20) + (119u << 23));  // 2^(E-8) * (1 + M/8)
}

}  // namespace rocmfp4
