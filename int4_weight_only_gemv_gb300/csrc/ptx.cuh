// ptx.cuh -- inline-PTX building blocks for the sm_103a kernels of the W4A16
// library: mbarriers, 1-D bulk (TMA) copies, cluster shared memory, and the
// register-level INT4 -> FP16 unpack.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace w4a16 {

// ---------------------------------------------------------------- addresses
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait that lets the thread sleep until the phase completes, for at most
// about `hint_ns` (the hardware may wake it earlier).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, for at most about
// `limit_ns` nanoseconds of wall time.  Returns false if the bound ran out.
// Each attempt sleeps until the phase completes (up to 1 ms), so a waiting
// warp takes no issue slots from the warps that are working.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- bulk copy
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar` with
// `bytes` of transaction count.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tiled bulk (TMA) copy global -> this CTA's shared memory through a
// tensor map (a __grid_constant__ kernel parameter), completing on `bar` with
// the box's bytes of transaction count.  x: innermost coordinate in elements
// (x * element size a multiple of 16 bytes), y: row.  Rows or columns past
// the tensor's extent are filled with zeros.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 3-D form of tma_load_2d: coordinates x (innermost, same alignment rule), y, z.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once (streamed weights).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data that other CTAs read soon after (kept at normal priority).
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- dependent launch
// Let the next kernel on the stream launch (it still waits for this one to
// finish before touching anything this one writes).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the previous kernel on the stream has completed and its writes
// are visible.  A no-op when the kernel was not launched as a dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// The two halves of cluster_sync, for a thread that has work to do in
// between.  Each thread alternates them (arrive, wait, arrive, ...).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Store to shared memory of another CTA of the cluster (a mapa'd address).
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------- shared loads
// Explicit shared-memory loads from 32-bit shared addresses (a pointer that
// went through integer arithmetic may otherwise be accessed generically).
__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint16_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void sts_u4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// 16 bytes through L1 (plain weak load).
__device__ __forceinline__ uint4 ld_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// 16 bytes through the read-only path (data constant for the kernel's life).
__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte asynchronous copy global -> this CTA's shared memory through the
// load path (cached in L2 only), waited for with cp_async_wait_all.  Both
// addresses 16-byte aligned.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Wait until every cp_async_16 this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Bring the 128-byte line holding p into this SM's L1 (no register result).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Acquire load at GPU scope: later loads of this thread see every write that
// was released (fence + atomic) before the value it returns was written.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------- unpack
// One packed word holds q[8j + i] in bits 4i..4i+3 (4-bit two's complement).
// With u = nibble ^ 8 = q + 8 in [0, 15], OR-ing u into the fraction of the
// fp16 constant 1024 (0x6400, unit in the last place 1) gives exactly
// 1024 + u; a nibble sitting at bits 4..7 of a 16-bit lane gives 1024 + 16 u.
// (w & mask) ^ (0x6400 | 8 << shift) does the mask, the XOR by 8 and the OR
// in one LOP3 (mask and constant exponent bits are disjoint).  For each
// 16-bit lane pair this yields, with v = w, v8 = w >> 8:
//   h0 = {1032 + q0, 1032 + q4}            from v  & 0x000F000F
//   h1 = {1152 + 16 q1, 1152 + 16 q5}      from v  & 0x00F000F0
//   h2 = {1032 + q2, 1032 + q6}            from v8 & 0x000F000F
//   h3 = {1152 + 16 q3, 1152 + 16 q7}      from v8 & 0x00F000F0
// All values are exact in fp16.
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) ^ c
  return d;
}

struct Unpacked {
  uint32_t h0, h1, h2, h3;
};

__device__ __forceinline__ Unpacked unpack_biased(uint32_t w) {
  const uint32_t w8 = w >> 8;
  Unpacked u;
  u.h0 = lop3_and_xor(w, 0x000F000Fu, 0x64086408u);
  u.h1 = lop3_and_xor(w, 0x00F000F0u, 0x64806480u);
  u.h2 = lop3_and_xor(w8, 0x000F000Fu, 0x64086408u);
  u.h3 = lop3_and_xor(w8, 0x00F000F0u, 0x64806480u);
  return u;
}

// For a tensor-core contraction: exact q in h0 = {q0,q4}, h2 = {q2,q6}, and
// h1 = {1152 + 16 q1, 1152 + 16 q5}, h3 = {1152 + 16 q3, 1152 + 16 q7} left
// as unpack_biased gives them (all exact in fp16).  Multiplied by x / 16,
// an odd lane gives q x + 72 x: the caller takes 72 x off once per group.
__device__ __forceinline__ Unpacked unpack_mma(uint32_t w) {
  Unpacked b = unpack_biased(w);
  const __half2 bias_lo = __half2half2(__ushort_as_half(0x6408));  // 1032
  __half2 t = __hsub2(*reinterpret_cast<__half2*>(&b.h0), bias_lo);
  b.h0 = *reinterpret_cast<uint32_t*>(&t);
  t = __hsub2(*reinterpret_cast<__half2*>(&b.h2), bias_lo);
  b.h2 = *reinterpret_cast<uint32_t*>(&t);
  return b;
}

// Exact q as fp16 pairs: {q0,q4}, {q1,q5}, {q2,q6}, {q3,q7}.
__device__ __forceinline__ Unpacked unpack_exact(uint32_t w) {
  Unpacked b = unpack_biased(w);
  const __half2 bias_lo = __half2half2(__ushort_as_half(0x6408));  // 1032
  const __half2 sixteenth = __half2half2(__ushort_as_half(0x2C00)); // 1/16
  const __half2 bias_hi = __half2half2(__ushort_as_half(0x5480));   // 72
  Unpacked q;
  __half2 t;
  t = __hsub2(*reinterpret_cast<__half2*>(&b.h0), bias_lo);
  q.h0 = *reinterpret_cast<uint32_t*>(&t);
  t = __hfma2(*reinterpret_cast<__half2*>(&b.h1), sixteenth, __hneg2(bias_hi));
  q.h1 = *reinterpret_cast<uint32_t*>(&t);
  t = __hsub2(*reinterpret_cast<__half2*>(&b.h2), bias_lo);
  q.h2 = *reinterpret_cast<uint32_t*>(&t);
  t = __hfma2(*reinterpret_cast<__half2*>(&b.h3), sixteenth, __hneg2(bias_hi));
  q.h3 = *reinterpret_cast<uint32_t*>(&t);
  return q;
}

// acc_lo += a.lo * b.lo ; acc_hi += a.hi * b.hi   (f16 x f16 products, f32 sums)
__device__ __forceinline__ void fma_f32_f16x2(float& acc_lo, float& acc_hi, uint32_t a,
                                              uint32_t b) {
  asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\t"
      "mov.b32 {b0, b1}, %3;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
      "fma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(a), "r"(b));
}

// Pairing of activations with the unpacked lanes of one word (8 halves
// x0..x7 loaded as uint4 {x1x0, x3x2, x5x4, x7x6}): {x0,x4} {x1,x5} {x2,x6} {x3,x7}.
struct XPairs {
  uint32_t p0, p1, p2, p3;
};

__device__ __forceinline__ XPairs pair_activations(uint4 v) {
  XPairs x;
  x.p0 = __byte_perm(v.x, v.z, 0x5410);
  x.p1 = __byte_perm(v.x, v.z, 0x7632);
  x.p2 = __byte_perm(v.y, v.w, 0x5410);
  x.p3 = __byte_perm(v.y, v.w, 0x7632);
  return x;
}

// GGUF Q4_K: sub-block j's 6-bit scale and minimum from a block's 12 packed
// bytes b (3 words, bytes 4-15 of the block): j < 4 in the low 6 bits of
// bytes j and j + 4; j >= 4 in the nibbles of byte j + 4 (scale low, minimum
// high) with their top two bits in bytes j - 4 (scale) and j (minimum).
__device__ __forceinline__ void q4k_scale_min(const uint32_t (&b)[3], int j, int& sc, int& m) {
  // word by selects, not by index: j may vary between threads
  auto byte = [&](int i) {
    const uint32_t w = i < 4 ? b[0] : (i < 8 ? b[1] : b[2]);
    return static_cast<int>((w >> (8 * (i & 3))) & 0xFFu);
  };
  if (j < 4) {
    sc = byte(j) & 63;
    m = byte(j + 4) & 63;
  } else {
    sc = (byte(j + 4) & 15) | ((byte(j - 4) >> 6) << 4);
    m = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
  }
}

__device__ __forceinline__ float half_lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

}  // namespace w4a16
