// Device-side building blocks shared by the kernels of libkvp (sm_103a):
// status recording, mbarrier waits with an iteration limit, bulk and tensor
// (TMA) copies into shared memory, the tcgen05 tensor-core primitives and the
// warp-level ldmatrix / mma.sync wrappers.
// Written from the PTX ISA's descriptions of these instructions.
#pragma once

#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "kvp.h"

#define KVP_DEV __device__ __forceinline__

namespace kvp {

constexpr int kPage = KVP_PAGE_TOKENS;
constexpr int32_t kNever = KVP_EXPIRE_NEVER;
// A wait on an mbarrier gives up after this much wall time (the %globaltimer
// clock); every wait in these kernels normally completes in microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

KVP_DEV void record_error(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Release/acquire fence at GPU scope, for message passing between CTAs: a
// writer orders its stores before its arrival on a counter, and the CTA that
// sees the final count orders its loads after it (no sequentially consistent
// fence is needed for that).
KVP_DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while the kernel before it on the stream is still
// running; it calls pdl_wait() before its first global memory access, which
// returns once that kernel has completed and its writes are visible (a no-op
// for a kernel launched without the attribute). pdl_launch_dependents() lets
// the next such kernel be scheduled without waiting for this one to exit.
KVP_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
KVP_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launches kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization allowed (the kernel must call pdl_wait() first).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  // a rejected launch (a configuration error, not a fault) is reported here and
  // taken off the runtime's last-error slot, so that the next call does not see it
  if (e != cudaSuccess) (void)cudaGetLastError();
  return e;
}

// launch_pdl with thread-block clusters of cluster_x CTAs (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                               unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  // a rejected launch (a configuration error, not a fault) is reported here and
  // taken off the runtime's last-error slot, so that the next call does not see it
  if (e != cudaSuccess) (void)cudaGetLastError();
  return e;
}

// Named barrier `id` (1..15) over n threads (a multiple of 32).
KVP_DEV void named_bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// The same, returning the OR of v over the n threads (every one of them must reach it).
KVP_DEV bool named_bar_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

KVP_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
KVP_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
KVP_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
KVP_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

KVP_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
KVP_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
KVP_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
KVP_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase of parity `parity` to complete. Gives up (returns
// false) after about limit_ns, as soon as *local_abort becomes nonzero, or
// once *status holds KVP_ERR_TIMEOUT (another CTA already gave up). The clock
// and the status word are only consulted every 1024 probes, so a short wait
// costs nothing but the barrier probes themselves.
KVP_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* local_abort = nullptr,
                       const volatile int32_t* status = nullptr, uint64_t limit_ns = kWaitLimitNs) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (local_abort != nullptr && *local_abort) return false;
    if ((i & 1023u) == 1023u) {
      if (status != nullptr && *status == KVP_ERR_TIMEOUT) return false;
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
KVP_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tensor-map (TMA) load of one box at coordinates (c0 = innermost, c1).
KVP_DEV void tma_load_2d(void* dst, const void* tmap, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
// The same box delivered to the same shared-memory offset in every CTA of the
// cluster named in cta_mask, each arrival counted on the mbarrier at `bar`'s
// offset in that CTA.
KVP_DEV void tma_load_2d_multicast(void* dst, const void* tmap, int c0, int c1, uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(cta_mask)
      : "memory");
}
// 3-D tensor-map (TMA) load of one box at coordinates (c0 = innermost, c1, c2).
KVP_DEV void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
KVP_DEV void tma_load_2d_hint(void* dst, const void* tmap, int c0, int c1, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
KVP_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
KVP_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
KVP_DEV void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Tensor memory allocation: one full warp executes these.
KVP_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
KVP_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"); }
KVP_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
KVP_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
KVP_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, issued by one thread.
KVP_DEV void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]: the A operand read from tensor memory
// (row m in lane m, two bf16 per 32-bit column, the lower k in the low half).
KVP_DEV void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same, always accumulating into d_tmem (no predicate to set per product).
KVP_DEV void umma_bf16_tmem_a_acc(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc) {
  asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc),
               "r"(idesc)
               : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completes.
KVP_DEV void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// The same, arriving on the mbarrier at `bar`'s offset in every CTA of the cluster named in cta_mask.
KVP_DEV void umma_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Thread-block clusters: this CTA's rank, and a barrier over every thread of
// every CTA of the cluster (release / acquire).
KVP_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
KVP_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, shape M x N.
constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// The same with the B operand MN-major (N contiguous in shared memory).
constexpr uint32_t kIdescBMnMajor = 1u << 16;

// Shared-memory matrix descriptor for a K-major tile whose rows are 128 bytes
// (64 bf16) stored with the 128-byte swizzle, 8-row groups 1024 bytes apart.
// The tile base must be 1024-byte aligned. Advancing K by 16 elements inside
// the row adds 32 bytes (2 in the >>4 address field).
KVP_DEV uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4)   // start address
         | (static_cast<uint64_t>(1) << 16)                 // leading byte offset (unused here)
         | (static_cast<uint64_t>(1024 >> 4) << 32)         // stride byte offset: 8 rows x 128 B
         | (static_cast<uint64_t>(1) << 46)                 // descriptor version
         | (static_cast<uint64_t>(2) << 61);                // 128-byte swizzle
}

// Shared-memory matrix descriptor for an MN-major operand with the 128-byte
// swizzle: each 1024-byte atom holds 8 consecutive k (rows of 128 bytes) of
// 64 consecutive m or n values; atoms along M/N lie mn_stride bytes apart,
// atoms along K (the next 8 k) k_stride bytes apart. Atoms 1024-byte aligned.
KVP_DEV uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t mn_stride, uint32_t k_stride) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4)            // start address
         | (static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16)  // leading byte offset
         | (static_cast<uint64_t>((k_stride >> 4) & 0x3FFFu) << 32)   // stride byte offset
         | (static_cast<uint64_t>(1) << 46)                           // descriptor version
         | (static_cast<uint64_t>(2) << 61);                          // 128-byte swizzle
}

// Loads 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per
// thread) and waits for them, in one asm block so no use can move above the wait.
KVP_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
KVP_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Stores 16, 8 or 4 consecutive 32-bit columns of this warp's 32 TMEM lanes.
KVP_DEV void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
KVP_DEV void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
KVP_DEV void tmem_st4(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
// Stores N (a multiple of 4) consecutive 32-bit columns of this warp's 32 TMEM lanes.
template <int N>
KVP_DEV void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N % 4 == 0, "columns in fours");
  int c = 0;
#pragma unroll
  for (; c + 16 <= N; c += 16) tmem_st16(taddr + c, r + c);
  if constexpr (N % 16 >= 8) {
    tmem_st8(taddr + c, r + c);
    c += 8;
  }
  if constexpr (N % 8 == 4) tmem_st4(taddr + c, r + c);
}
// Loads N (a multiple of 16) consecutive fp32 columns of this warp's 32 TMEM lanes, waiting for each part.
template <int N>
KVP_DEV void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  static_assert(N % 16 == 0, "columns in sixteens");
  int c = 0;
#pragma unroll
  for (; c + 32 <= N; c += 32) tmem_ld32(taddr + c, *reinterpret_cast<float(*)[32]>(&v[c]));
#pragma unroll
  for (; c + 16 <= N; c += 16) tmem_ld16(taddr + c, *reinterpret_cast<float(*)[16]>(&v[c]));
}

// Stores 32 consecutive 32-bit columns of this warp's 32 TMEM lanes (one row
// per thread); tmem_st_wait() waits for the stores issued so far.
KVP_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
KVP_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- warp-level tensor-core products
// ldmatrix: four 8x8 b16 matrices from shared memory, the row addresses given
// by lanes 8i..8i+7 for matrix i (.trans: each matrix transposed on the way).
KVP_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
KVP_DEV void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
// d += A B, A 16 x 16 (row), B 16 x 8 (col), fp16 in, fp32 accumulate
KVP_DEV void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// d += A B, A 16 x 16 (row), B 16 x 8 (col), bf16 in, fp32 accumulate
KVP_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                            uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x by the PTX instruction ex2.approx.ftz.f32 (the special-function unit's
// base-2 exponential, within a few units in the last place; subnormal results
// flush to zero and 2^-inf = 0).
KVP_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- E4M3 conversions
// Two E4M3 codes (the first in the low byte of `two`) to two fp16 values (the
// first in the low half), exactly: every E4M3 value is an fp16 value. One PTX
// conversion instruction (cvt.rn.f16x2.e4m3x2).
KVP_DEV uint32_t cvt_e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(two & 0xFFFFu)));
  return r;
}
// Two fp32 values to E4M3 codes, rounded to nearest (ties to even) and
// saturated to +-448, `lo` in the low byte. One PTX conversion instruction
// (cvt.rn.satfinite.e4m3x2.f32, whose first source fills the high byte).
KVP_DEV uint32_t cvt_f32x2_to_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------- bf16 helpers
KVP_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
KVP_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- host: TMA descriptors
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] (row stride ld elements) read in boxes of
// box_rows x box_cols with the 128-byte swizzle; zero fill outside the matrix.
inline bool make_tmap_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                           int box_cols) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A byte matrix [rows, row_bytes] (row_bytes 64 or 128, rows packed) whose
// box is box_rows whole rows, landing in shared memory with the swizzle of its
// row width: 16-byte chunk c of box row r at chunk c ^ (r & 7) of a 128-byte
// row, or c ^ ((r >> 1) & 3) of a 64-byte row (the destination aligned to
// 1024 or 512 bytes).
inline bool make_tmap_u8_rows(CUtensorMap* m, const void* base, int64_t rows, int row_bytes, int box_rows) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr || (row_bytes != 64 && row_bytes != 128) || rows <= 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major bf16 matrix [rows, cols] (cols a multiple of 64, row stride ld
// elements) seen as [rows][cols / 64][64]: one box is box_rows consecutive rows
// x every 64-column group, landing in shared memory as cols / 64 boxes of
// box_rows x 128 bytes one after another (group-major), each with the 128-byte
// swizzle. Dimension 1 (rows) has the larger stride; dimension 2 (the 64-column
// group) steps 128 bytes.
inline bool make_tmap_bf16_groups(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld,
                                  int box_rows) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr || cols % 64 != 0 || cols / 64 > 256) return false;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(cols / 64)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kvp
