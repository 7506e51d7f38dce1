// common.cuh -- shared device helpers for the sm_103a kernels: bf16
// conversion, Philox4x32-10, mbarrier / TMA / tcgen05 inline PTX wrappers
// and bounded waits.  Every spin-wait here gives up after a time limit and
// reports through a device error word instead of hanging the GPU.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wsnf4.h"

#define WS_DEVINL __device__ __forceinline__

namespace ws {

// ---- error word -------------------------------------------------------------
// Bit flags a kernel ORs into the library's device error word.
// (The public bits in wsnf4.h: WS_DERR_PIPELINE_MASK covers bits 0-5,
// WS_DERR_BAD_CONFIG is bit 6, WS_DERR_TIMEOUT_PEER bit 7.)
enum : uint32_t {
  DERR_TIMEOUT_FULL = 1u << 0,
  DERR_TIMEOUT_EMPTY = 1u << 1,
  DERR_TIMEOUT_BFULL = 1u << 2,
  DERR_TIMEOUT_BEMPTY = 1u << 3,
  DERR_TIMEOUT_ACC = 1u << 4,
  DERR_TIMEOUT_DRAIN = 1u << 5,
  DERR_BAD_CONFIG = WS_DERR_BAD_CONFIG,
  DERR_TIMEOUT_PEER = WS_DERR_TIMEOUT_PEER,
};
static_assert((DERR_TIMEOUT_FULL | DERR_TIMEOUT_EMPTY | DERR_TIMEOUT_BFULL | DERR_TIMEOUT_BEMPTY |
               DERR_TIMEOUT_ACC | DERR_TIMEOUT_DRAIN) == WS_DERR_PIPELINE_MASK,
              "device error bits");

#if defined(WS_GEMM_TU) || defined(WS_ATTN_TU)
// Device error word of a translation unit with spin-waits (the GEMM unit and
// the attention unit each own one); ws_device_error reads and clears both.
static __device__ uint32_t g_dev_error = 0;
#define WS_HAS_WAITS 1
#endif

// Wall-clock limit of one wait (ns).  Pipeline waits in these kernels are
// microseconds long; a second means the pipeline is broken.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

WS_DEVINL uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- bf16 ----------------------------------------------------------------------
WS_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  // cvt.rn.bf16x2.f32 d, a, b puts a in the upper half and b in the lower.
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
WS_DEVINL float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
WS_DEVINL float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
WS_DEVINL float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
WS_DEVINL uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ---- Philox4x32-10 ---------------------------------------------------------------
// Counter-based generator of Salmon et al. (SC'11): ten rounds of two 32x32
// multiplies, the key bumped by the Weyl increments between rounds.
struct u32x4 {
  uint32_t x, y, z, w;
};
WS_DEVINL u32x4 philox4x32_10(u32x4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = u32x4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Keep mask of 4 consecutive elements e0..e0+3 (e0 % 4 == 0) of one linear's
// dropout input, as 4 bits (bit i <-> element e0 + i).
// Counter = (e >> 2, linear | microbatch << 8, layer, step); key = seed.
struct DropKey {
  uint32_t k0, k1;   // seed low / high words
  uint32_t c1, c2, c3;
  uint32_t thresh;   // keep <=> word >= thresh  (thresh_is_max: drop all)
  uint32_t drop_all; // p == 1 (threshold 2^32)
  const uint32_t* step_dev;  // when set, the step word c3 is read from here
};
// Resolve the step word once per thread (device-resident step for graphs).
WS_DEVINL void resolve_step(DropKey& k) {
  if (k.step_dev) k.c3 = *k.step_dev;
}
WS_DEVINL uint32_t keep4(const DropKey& k, uint64_t e0) {
  if (k.drop_all) return 0u;
  const u32x4 r = philox4x32_10(u32x4{(uint32_t)(e0 >> 2), k.c1, k.c2, k.c3}, k.k0, k.k1);
  return (uint32_t)(r.x >= k.thresh) | ((uint32_t)(r.y >= k.thresh) << 1) |
         ((uint32_t)(r.z >= k.thresh) << 2) | ((uint32_t)(r.w >= k.thresh) << 3);
}

// ---- shared-memory address ---------------------------------------------------------
WS_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
WS_DEVINL void sts128(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}
// One 32-byte global load (p 32-byte aligned).
WS_DEVINL void ld_global_v8(const void* p, uint32_t* r) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "l"(p)
               : "memory");
}
// One 32-byte global store (p 32-byte aligned).
WS_DEVINL void st_global_v8(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                            uint32_t f, uint32_t g, uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a), "r"(b),
               "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
               : "memory");
}

// ---- mbarrier --------------------------------------------------------------------------
WS_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
WS_DEVINL void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
WS_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
      : "memory");
}
WS_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
WS_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
#ifdef WS_HAS_WAITS
// Bounded wait for the phase with the given parity to complete.  Returns
// false (and records `why` in the device error word) on timeout.
WS_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t why) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u && globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&g_dev_error, why);
      return false;
    }
  }
}

// Same, for waits expected to last a whole main loop (epilogue warps): poll
// with a short sleep so the waiting warps leave issue slots to the producers.
WS_DEVINL bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, uint32_t why) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(200);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u && globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&g_dev_error, why);
      return false;
    }
  }
}
#endif

// ---- cross-CTA flags ---------------------------------------------------------------------
WS_DEVINL uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
#ifdef WS_HAS_WAITS
// Bounded wait (acquire) for a cross-CTA word to hold `expect`: polls with a
// short sleep; after limit_ns of wall-clock time it records `why` in the
// device error word and returns false.
WS_DEVINL bool wait_flag_bounded(const uint32_t* f, uint32_t expect, uint64_t limit_ns,
                                 uint32_t why) {
  if (ld_acquire_gpu(f) == expect) return true;
  const uint64_t t0 = globaltimer();
  while (ld_acquire_gpu(f) != expect) {
    __nanosleep(128);
    if (globaltimer() - t0 > limit_ns) {
      atomicOr(&g_dev_error, why);
      return false;
    }
  }
  return true;
}
#endif
WS_DEVINL void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- fences ----------------------------------------------------------------------------
// Make generic-proxy shared-memory writes visible to the async proxy
// (tensor cores, TMA) before signalling a barrier.
WS_DEVINL void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA ---------------------------------------------------------------------------------
WS_DEVINL void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
WS_DEVINL void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x,
                           int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned addresses, size a
// multiple of 16), completing as transaction bytes on a local mbarrier.
WS_DEVINL void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- tcgen05 -------------------------------------------------------------------------------
WS_DEVINL void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
WS_DEVINL void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
WS_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
WS_DEVINL void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
WS_DEVINL void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, f32 acc).
WS_DEVINL void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when all previously issued tcgen05 ops of this thread
// have completed.
WS_DEVINL void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: lane i of the warp receives row
// (32*(warp%4) + i), columns [col, col+32).
WS_DEVINL void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
WS_DEVINL void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
WS_DEVINL void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive 32-bit columns back into TMEM (same layout as
// tmem_ld_32x32b_x16).
WS_DEVINL void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
WS_DEVINL void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (>> 4), fixed version bits 46-48 = 0b001, 128-byte
// swizzle (layout type 2 in bits 61-63).
WS_DEVINL uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, A
// K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), N >> 3 at bit 17,
// M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

WS_DEVINL uint32_t warp_id() { return threadIdx.x >> 5; }
WS_DEVINL uint32_t lane_id() { return threadIdx.x & 31; }
WS_DEVINL bool elect_lane0() { return lane_id() == 0; }

// ---- thread-block clusters ------------------------------------------------------------
WS_DEVINL uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
WS_DEVINL uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
WS_DEVINL uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
WS_DEVINL void st_cluster_v4(uint32_t caddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's earlier writes at cluster scope.
WS_DEVINL void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar)
               : "memory");
}
// The same arrival with release at CTA scope (the instruction's default
// semantics): orders this CTA's earlier shared-memory writes and completed
// tensor-memory accesses before it, which is all a pair partner needs when
// the data handed over lies in this CTA's own shared or tensor memory.  A
// cluster-scope release costs about as much as a pipeline step of the
// dequant GEMM (its forwarding thread's release alone held the 256-wide
// steps at 0.8 us).
WS_DEVINL void mbar_arrive_remote(uint32_t cbar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
WS_DEVINL bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Commit: the mbarrier at this offset in every CTA of `mask` receives one
// arrival once this thread's earlier tcgen05 operations have completed.
WS_DEVINL void tc_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}
// Copy `bytes` of this CTA's shared memory to a shared::cluster address in
// another CTA of the cluster; completion is signalled as transaction bytes
// on that CTA's mbarrier (cluster address cbar).
WS_DEVINL void bulk_copy_to_peer(uint32_t cdst, const void* src, uint32_t bytes, uint32_t cbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(cdst), "r"(smem_u32(src)), "r"(bytes), "r"(cbar)
      : "memory");
}
// ---- CTA pairs: one tensor-core operation across both CTAs of a cluster of two ---------
// Every tcgen05 instruction of a kernel uses the same CTA group, so a kernel
// that issues pair MMAs allocates, commits and frees through these.
// Both CTAs allocate (the same columns in each CTA's tensor memory).
WS_DEVINL void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
WS_DEVINL void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
WS_DEVINL void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Issued by the even CTA only: M = 256 rows, the first 128 from the even
// CTA's A operand and the next 128 from the odd CTA's (same shared-memory
// offset in each); B's first N/2 columns from the even CTA, the rest from
// the odd one; D lands in each CTA's tensor memory at the same address.
WS_DEVINL void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                               uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
WS_DEVINL void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
WS_DEVINL void tc_commit_pair_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}
// Tile load into this CTA's shared memory whose completion bytes go to an
// mbarrier of either CTA of the pair (cluster address cbar).
WS_DEVINL void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t cbar, int32_t x,
                                int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(cbar), "r"(x), "r"(y)
      : "memory");
}

WS_DEVINL void fence_proxy_async_cluster() {
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}
WS_DEVINL void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

#ifdef WS_HAS_WAITS
// Same, acquiring at cluster scope (arrivals released by the other CTA of a pair).
WS_DEVINL bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t why) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 255u) == 0u && globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&g_dev_error, why);
      return false;
    }
  }
}

#endif

// ---- programmatic dependent launch ----------------------------------------------------
// Kernels are launched with programmatic stream serialization: the next
// kernel in the stream may be scheduled while this one still runs, does its
// own setup (barriers, tensor memory, descriptors), and waits here before
// its first access to global memory that an earlier kernel writes or reads.
// Once past the wait every earlier kernel of the stream has completed and
// its writes are visible.  Without that launch attribute the wait returns
// at once.
WS_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allows the next kernel of the stream to be scheduled (it still waits for
// this grid to complete before touching data).
WS_DEVINL void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier among `nthreads` threads (id 1..15; id 0 is __syncthreads).
WS_DEVINL void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Host: launch with programmatic stream serialization (unless
// WS_NF4_PDL=0).  Every kernel launched this way calls pdl_wait() before its
// first dependent global access.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace ws
