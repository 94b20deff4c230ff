// moe_device.cuh -- device helpers shared by the sm_103a kernels of libmoe.so:
// mbarrier / bulk-copy (TMA) wrappers in inline PTX, warp utilities, and the
// launcher declarations the C-ABI layer calls.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// Upper bound on polls of one mbarrier phase before a kernel gives up, sets
// MOE_ERR_DEVICE_TIMEOUT and returns. try_wait itself suspends for a bounded
// time per poll, so this bounds the wait to seconds, far above any legitimate
// copy latency.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
    }
    return false;
}

// Global -> shared bulk copy; completion is counted in bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Shared -> global bulk copy, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte read-only load that skips L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch. Every kernel of the path is launched with
// programmatic stream serialisation: it may be scheduled while the previous
// kernel on the stream is still running. It waits for that kernel (and so,
// transitively, everything before it) to complete and flush before its first
// global-memory access, then lets the next kernel be scheduled.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Record a device-side status in the caller's error word (any writer wins;
// all writers of one launch write codes, never 0).
__device__ __forceinline__ void raise_error(int32_t* err, int32_t code) {
    if (err) *reinterpret_cast<volatile int32_t*>(err) = code;
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Balanced split of n items over b parts, the first n % b parts one larger.
__host__ __device__ __forceinline__ void split_range(int64_t n, int64_t b, int64_t i, int64_t* begin,
                                                     int64_t* end) {
    const int64_t q = n / b, r = n % b;
    const int64_t s = i * q + (i < r ? i : r);
    *begin = s;
    *end = s + q + (i < r ? 1 : 0);
}

// ---------------------------------------------------------------------------
// Device-side phase profile (profile builds only, -DMOE_PROFILE; the default
// build compiles these macros to nothing). An instrumented kernel calls
// MOE_PROF_BEGIN(kernel) once, MOE_STAMP(p) at the end of phase p and
// MOE_PROF_END() before it returns. Thread 0 of CTA b keeps the stamps in
// shared memory while the kernel runs (a global store would make the next
// cluster barrier's release wait for it) and writes them at the end to row
//   slots[(kernel * kProfCtas + b) * kProfPhases ...]
// of the array attached with moe_profile_attach: slot 0 = %globaltimer (ns) at
// MOE_PROF_BEGIN, slot p = clock64 cycles from MOE_PROF_BEGIN to the end of
// phase p (0 if not reached), and the last slot 1 + the SM the CTA ran on
// (%smid). CTAs at or beyond kProfCtas record nothing.
// Loop phases that repeat inside a CTA (the int8 consumer's per-token steps)
// are summed in registers by one thread and written with MOE_PROF_PUT, the
// start stamp alone then being published with MOE_PROF_END_N(1).
#ifdef MOE_PROFILE
constexpr int kProfKernels = MOE_PROF_KERNELS;
constexpr int kProfCtas = MOE_PROF_CTAS;
constexpr int kProfPhases = MOE_PROF_PHASES;
enum ProfKernel { kProfLayout = 0, kProfNotify = 1, kProfDispatch = 2, kProfDispatchInt8 = 3, kProfCombine = 4,
                  kProfFused = 5, kProfNotifyExpert = 6, kProfExpertCount = 7 };
// One copy per translation unit, set by that unit's prof_attach_* function.
static __device__ unsigned long long* g_prof_slots;

__device__ __forceinline__ unsigned long long prof_globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned long long prof_smid() {
    unsigned int v;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
    return v;
}
__device__ __forceinline__ unsigned long long* prof_row(int kernel) {
    unsigned long long* p = g_prof_slots;
    if (p == nullptr || blockIdx.x >= static_cast<unsigned>(kProfCtas)) return nullptr;
    return p + (static_cast<size_t>(kernel) * kProfCtas + blockIdx.x) * kProfPhases;
}
#define MOE_PROF_BEGIN(kernel)                                                        \
    __shared__ unsigned long long moe_prof_sm_[kProfPhases];                          \
    unsigned long long* const moe_prof_row_ = ::moe::prof_row(kernel);                \
    const long long moe_prof_c0_ = clock64();                                         \
    if (threadIdx.x == 0) {                                                           \
        moe_prof_sm_[0] = ::moe::prof_globaltimer();                                  \
        for (int moe_i_ = 1; moe_i_ < kProfPhases; ++moe_i_) moe_prof_sm_[moe_i_] = 0; \
        moe_prof_sm_[kProfPhases - 1] = ::moe::prof_smid() + 1;                         \
    }
#define MOE_STAMP(phase)                                                              \
    do {                                                                              \
        if (threadIdx.x == 0)                                                         \
            moe_prof_sm_[(phase)] = static_cast<unsigned long long>(clock64() - moe_prof_c0_); \
    } while (0)
#define MOE_PROF_END_N(n)                                                             \
    do {                                                                              \
        if (moe_prof_row_ && threadIdx.x == 0)                                        \
        {                                                                             \
            for (int moe_i_ = 0; moe_i_ < (n); ++moe_i_) moe_prof_row_[moe_i_] = moe_prof_sm_[moe_i_]; \
            moe_prof_row_[kProfPhases - 1] = moe_prof_sm_[kProfPhases - 1];           \
        }                                                                             \
    } while (0)
#define MOE_PROF_END() MOE_PROF_END_N(kProfPhases)
#define MOE_PROF_CLOCK() clock64()
#define MOE_PROF_PUT(phase, value)                                                    \
    do {                                                                              \
        if (moe_prof_row_) moe_prof_row_[(phase)] = static_cast<unsigned long long>(value); \
    } while (0)
// Defines prof_attach_<unit>(), which points this unit's kernels at `slots`.
#define MOE_PROFILE_UNIT(unit)                                                      \
    cudaError_t prof_attach_##unit(void* slots) {                                  \
        unsigned long long* p = static_cast<unsigned long long*>(slots);           \
        return cudaMemcpyToSymbol(g_prof_slots, &p, sizeof(p));                    \
    }
cudaError_t prof_attach_layout(void*);
cudaError_t prof_attach_notify(void*);
cudaError_t prof_attach_dispatch(void*);
cudaError_t prof_attach_combine(void*);
cudaError_t prof_attach_fused(void*);
cudaError_t prof_attach_expert(void*);
#else
#define MOE_PROF_BEGIN(kernel) \
    do {                       \
    } while (0)
#define MOE_PROF_END() \
    do {               \
    } while (0)
#define MOE_PROF_END_N(n) \
    do {                  \
    } while (0)
#define MOE_STAMP(phase) \
    do {                 \
    } while (0)
#define MOE_PROF_CLOCK() 0ll
#define MOE_PROF_PUT(phase, value) \
    do {                           \
    } while (0)
#define MOE_PROFILE_UNIT(unit)
#endif

// ---------------------------------------------------------------------------
// Launchers (defined in layout.cu / notify.cu / dispatch.cu / combine.cu).
// Shapes are validated by the C-ABI layer before these run.

struct LayoutPlan {
    int cluster;   // CTAs per source rank (before the residency check)
    int threads;   // tokens per block pass (one per thread)
    size_t smem;
    int64_t scratch_bytes;  // one out-of-range flag per source rank
};
LayoutPlan layout_plan(const moe_shape& s);
cudaError_t launch_layout(const moe_shape& s, const int32_t* topk_idx, int32_t* ntpr, int32_t* ntpe,
                          uint8_t* itr, uint32_t* bits, int32_t* err, void* scratch,
                          cudaStream_t stream);

int64_t notify_scratch_bytes(const moe_shape& s);
cudaError_t launch_notify(const moe_shape& s, const int32_t* ntpr, const int32_t* ntpe,
                          const uint8_t* itr, int32_t* rpm, int32_t* cpm, int32_t* rcpm,
                          int32_t* nrt, int32_t* nrtpe, int32_t* reo, int32_t* send_head,
                          int64_t* part_row_base, void* scratch, cudaStream_t stream);

struct DispatchArgs {
    int32_t P, E, K, H, epr;
    int64_t S, T;
    const uint16_t* x;
    const int32_t* topk_idx;
    const float* topk_weights;
    const int32_t* send_head;
    const int64_t* part_row_base;
    uint8_t* arena;
    int64_t arena_rows;
    int64_t stride;
    int64_t scale_off;
    int64_t triple_off;
    int32_t* recv_src_idx;
    int32_t* recv_topk_idx;
    float* recv_topk_weights;
    int32_t* err;
    int32_t stages;
    uint32_t row_bytes;  // bf16 bytes of one source row, H * 2
    // Expert-major layout only: one slot per (token, k).
    const int32_t* slot_row;  // [S, K] row inside the destination rank's partition, or -1
    float* recv_weight;       // [rows] the slot's Top-K weight (may be NULL)
};
cudaError_t launch_dispatch(const moe_shape& s, DispatchArgs a, cudaStream_t stream);
cudaError_t launch_dispatch_expert(const moe_shape& s, DispatchArgs a, cudaStream_t stream);

struct CombineArgs {
    int32_t P, E, K, H, epr;
    int64_t S;
    const uint8_t* y;
    int64_t y_stride;
    const int64_t* part_row_base;
    int64_t arena_rows;
    const int32_t* send_head;
    const int32_t* topk_idx;
    const float* topk_weights;
    uint16_t* out;
    int32_t* err;
    const int32_t* slot_row;  // expert-major layout only
};
cudaError_t launch_combine(const moe_shape& s, CombineArgs a, cudaStream_t stream);
cudaError_t launch_combine_expert(const moe_shape& s, CombineArgs a, cudaStream_t stream);

int64_t notify_expert_scratch_bytes(const moe_shape& s);
cudaError_t launch_notify_expert(const moe_shape& s, const int32_t* topk_idx, const int32_t* nrtpe,
                                 const int32_t* reo, int32_t* slot_row, int64_t* expert_part_base,
                                 void* scratch, cudaStream_t stream);

cudaError_t launch_pad(const moe_shape& s, const int32_t* nrt, const int64_t* prb, uint8_t* arena,
                       int64_t arena_rows, int32_t* src_idx, int32_t* tk_idx, float* tk_w,
                       cudaStream_t stream);

bool fused_supported(const moe_shape& s);
// Test hook behind moe_test_fused_barrier (this host thread's next fused launch).
void arm_fused_barrier_test(uint32_t spin_limit, int64_t skip_cta);
int64_t fused_scratch_bytes(const moe_shape& s);
cudaError_t launch_fused(const moe_shape& s, const uint16_t* x, const int32_t* topk_idx, const float* topk_weights,
                         int32_t* ntpr, int32_t* ntpe, uint8_t* itr, uint32_t* bits, int32_t* rpm, int32_t* cpm,
                         int32_t* rcpm, int32_t* nrt, int32_t* nrtpe, int32_t* reo, int32_t* send_head,
                         int64_t* part_row_base, const DispatchArgs& d, int32_t* err, void* scratch,
                         cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();
// Opt-in shared memory per block of the current device (cached).
int device_optin_smem();
// Shared memory of one SM (all its CTAs together), per current device.
int device_sm_smem();
// Allow `fn` `smem` bytes of dynamic shared memory on the current device and,
// if per_sm is given, return its resident blocks per SM for (threads, smem).
// Both are cached per (kernel, device).
cudaError_t prepare_kernel(const void* fn, size_t smem, int threads, int* per_sm);
// Static shared memory of `fn` (cached), or -1.
int kernel_static_smem(const void* fn);

// Launch `kernel` on `stream` with programmatic stream serialisation (see
// pdl_wait_then_release); the kernel must call pdl_wait_then_release before
// touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl for a kernel whose blocks form thread-block clusters of
// `cluster` CTAs along x (grid a multiple of cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                               unsigned cluster, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Largest cluster size c in {want, want/2, ..., 1} for which clusters of c
// CTAs of `fn` (threads, smem) can be resident on the current device; cached
// per (kernel, device, want, threads, smem).
int cluster_size_for(const void* fn, int want, int threads, size_t smem);

// ---------------------------------------------------------------------------
// Thread-block cluster helpers (distributed shared memory).

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Index of this CTA's cluster along x (the grid is clusters of CTAs along x).
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Full cluster barrier: release this thread's prior memory operations
// (shared and distributed shared) and acquire the other CTAs'.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Split form of the barrier: arrive now, wait later (the CTA's shared memory
// must stay valid until every peer has passed its wait).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of `p` (a shared-memory location of this CTA) in the shared
// memory of cluster CTA `rank`, as a shared::cluster address.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(p)), "r"(rank));
    return out;
}

__device__ __forceinline__ int32_t ld_cluster_s32(uint32_t addr) {
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

}  // namespace moe
