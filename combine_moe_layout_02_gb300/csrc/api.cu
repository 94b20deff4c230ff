// api.cu -- the C ABI of libmoe.so (declared in include/moe.h): host-side
// validation, scratch sizing and the launches on the caller's stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "moe.h"
#include "moe_device.cuh"

namespace moe {

namespace {

// A device attribute, cached per device (0 = not read yet). Threads that race
// on a first read store the same value.
int cached_attribute(std::atomic<int> (&cache)[64], cudaDeviceAttr attr, int fallback) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fallback;
    const bool slot = dev >= 0 && dev < 64;
    if (slot) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, attr, dev) != cudaSuccess || n < 1) return fallback;
    if (slot) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

std::atomic<int> g_sm_count[64];
std::atomic<int> g_optin_smem[64];
std::atomic<int> g_sm_smem[64];

}  // namespace

int device_sm_count() { return cached_attribute(g_sm_count, cudaDevAttrMultiProcessorCount, 1); }

int device_optin_smem() {
    return cached_attribute(g_optin_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, 48 * 1024);
}

int device_sm_smem() {
    return cached_attribute(g_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, 64 * 1024);
}

namespace {

// Per (kernel, device): the dynamic shared memory the kernel has been allowed
// so far, its static shared memory, and the last occupancy query. Launches
// then skip repeated runtime queries; the allowance only ever grows, so a
// concurrent launch with a smaller request stays valid.
struct KernelEntry {
    const void* fn;
    int dev, smem_allowed, occ_threads, occ, static_smem;
    size_t occ_smem;
};
std::mutex g_kernel_mu;
KernelEntry g_kernels[256];
int g_nkernels = 0;

KernelEntry* kernel_entry(const void* fn, int dev) {  // g_kernel_mu held
    for (int i = 0; i < g_nkernels; ++i)
        if (g_kernels[i].fn == fn && g_kernels[i].dev == dev) return &g_kernels[i];
    if (g_nkernels == 256) return nullptr;
    g_kernels[g_nkernels] = KernelEntry{fn, dev, 0, -1, 0, -1, 0};
    return &g_kernels[g_nkernels++];
}

}  // namespace

cudaError_t prepare_kernel(const void* fn, size_t smem, int threads, int* per_sm) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_kernel_mu);
    KernelEntry* k = kernel_entry(fn, dev);
    if (k == nullptr || static_cast<int64_t>(smem) > k->smem_allowed) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (k) k->smem_allowed = static_cast<int>(smem);
    }
    if (per_sm) {
        if (k == nullptr || k->occ_threads != threads || k->occ_smem != smem) {
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
            if (e != cudaSuccess) return e;
            if (k) {
                k->occ_threads = threads;
                k->occ_smem = smem;
                k->occ = n;
            }
            *per_sm = n;
        } else {
            *per_sm = k->occ;
        }
    }
    return cudaSuccess;
}

namespace {

struct ClusterEntry {
    const void* fn;
    int dev, want, threads, result;
    size_t smem;
};
ClusterEntry g_clusters[256];
int g_nclusters = 0;

}  // namespace

int cluster_size_for(const void* fn, int want_in, int threads, size_t smem) {
    int want = want_in;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    {
        std::lock_guard<std::mutex> lock(g_kernel_mu);
        for (int i = 0; i < g_nclusters; ++i) {
            const ClusterEntry& c = g_clusters[i];
            if (c.fn == fn && c.dev == dev && c.want == want_in && c.threads == threads && c.smem == smem)
                return c.result;
        }
    }
    int result = -1;
    // Clusters above the portable 8 CTAs must be allowed per kernel.
    if (want > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        want = 8;
    }
    for (int c = want; c >= 1; c /= 2) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(c));
        cfg.blockDim = dim3(static_cast<unsigned>(threads));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(c);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n > 0) {
            result = c;
            break;
        }
        cudaGetLastError();  // clear a refusal of this size before trying the next
    }
    std::lock_guard<std::mutex> lock(g_kernel_mu);
    if (result > 0 && g_nclusters < 256) g_clusters[g_nclusters++] = ClusterEntry{fn, dev, want_in, threads, result, smem};
    return result;
}

int kernel_static_smem(const void* fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lock(g_kernel_mu);
    KernelEntry* k = kernel_entry(fn, dev);
    if (k && k->static_smem >= 0) return k->static_smem;
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return -1;
    if (k) k->static_smem = static_cast<int>(fa.sharedSizeBytes);
    return static_cast<int>(fa.sharedSizeBytes);
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Required array: non-NULL (unless it would hold no element) and aligned.
bool ok_ptr(const void* p, int64_t elements, uintptr_t align) {
    if (elements == 0) return p == nullptr || aligned(p, align);
    return p != nullptr && aligned(p, align);
}

// Optional array: NULL, or aligned.
bool ok_opt(const void* p, uintptr_t align) { return p == nullptr || aligned(p, align); }

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int32_t status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_TOPK_OUT_OF_RANGE: return "MOE_ERR_TOPK_OUT_OF_RANGE";
        case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
        case MOE_ERR_INCONSISTENT: return "MOE_ERR_INCONSISTENT";
        default: return "MOE_ERR_UNKNOWN";
    }
}

moe_status moe_check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->P < 1 || s->E < 1 || s->S < 0 || s->K < 1 || s->H < 1) return MOE_ERR_INVALID_ARG;
    if (s->num_channels < 1 || s->expert_alignment < 1) return MOE_ERR_INVALID_ARG;
    if (s->quant != 0 && s->quant != 1) return MOE_ERR_INVALID_ARG;
    if (s->E % s->P != 0 || s->S % s->P != 0) return MOE_ERR_INVALID_ARG;
    if (s->P > MOE_MAX_RANKS || s->E > MOE_MAX_EXPERTS || s->K > MOE_MAX_TOPK || s->H > MOE_MAX_HIDDEN)
        return MOE_ERR_UNSUPPORTED;
    if (s->num_channels > 4096) return MOE_ERR_UNSUPPORTED;
    if (s->H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (s->quant && s->H % 16 != 0) return MOE_ERR_INVALID_ARG;
    // Row counts and offsets are int32: the expert-major bound on one rank's
    // rows, S*K + E*(expert_alignment-1), must fit.
    if (static_cast<int64_t>(s->S) * s->K + static_cast<int64_t>(s->E) * (s->expert_alignment - 1) > INT32_MAX)
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int64_t moe_slot_stride(int32_t H, int32_t quant) {
    if (H < 1) return -1;
    const int64_t elt = quant ? 1 : 2;
    return round_up(round_up(static_cast<int64_t>(H) * elt, 32) + 44, 512);
}

int64_t moe_scratch_bytes(const moe_shape* s) {
    if (moe_check_shape(s) != MOE_OK) return -1;
    const int64_t a = layout_plan(*s).scratch_bytes;
    const int64_t b = notify_scratch_bytes(*s);
    const int64_t c = notify_expert_scratch_bytes(*s);
    const int64_t f = fused_supported(*s) ? fused_scratch_bytes(*s) : 0;
    int64_t m = a > b ? a : b;
    m = m > c ? m : c;
    m = m > f ? m : f;
    return m > 256 ? m : 256;
}

int64_t moe_max_expert_rows(const moe_shape* s) {
    if (moe_check_shape(s) != MOE_OK) return -1;
    return static_cast<int64_t>(s->S) * s->K + static_cast<int64_t>(s->E) * (s->expert_alignment - 1);
}

int64_t moe_max_recv_rows(const moe_shape* s) {
    if (moe_check_shape(s) != MOE_OK) return -1;
    const int64_t m = s->K < s->P ? s->K : s->P;
    return static_cast<int64_t>(s->S) * m;
}

moe_status moe_layout(const moe_shape* shape, const int32_t* topk_idx, int32_t* num_tokens_per_rank,
                      int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                      uint32_t* is_token_in_rank_bits, int32_t* err, void* scratch,
                      int64_t scratch_bytes, void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if (!ok_ptr(topk_idx, S * s.K, 16) || !ok_ptr(num_tokens_per_rank, 1, 16) ||
        !ok_ptr(num_tokens_per_expert, 1, 16) || !ok_ptr(is_token_in_rank, S * s.P, 16) ||
        !ok_opt(is_token_in_rank_bits, 16) || !ok_opt(err, 4) || !ok_ptr(scratch, 1, 256))
        return MOE_ERR_INVALID_ARG;
    if (scratch_bytes < moe_scratch_bytes(shape)) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_layout(s, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                                   is_token_in_rank, is_token_in_rank_bits, err, scratch,
                                   static_cast<cudaStream_t>(stream)));
}

moe_status moe_notify(const moe_shape* shape, const int32_t* num_tokens_per_rank,
                      const int32_t* num_tokens_per_expert, const uint8_t* is_token_in_rank,
                      int32_t* rank_prefix_matrix, int32_t* channel_prefix_matrix,
                      int32_t* recv_channel_prefix_matrix, int32_t* num_recv_tokens,
                      int32_t* num_recv_tokens_per_expert, int32_t* recv_expert_offset,
                      int32_t* send_head, int64_t* part_row_base, void* scratch,
                      int64_t scratch_bytes, void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if (!ok_ptr(num_tokens_per_rank, 1, 16) || !ok_ptr(num_tokens_per_expert, 1, 16) ||
        !ok_ptr(is_token_in_rank, S * s.P, 16) || !ok_ptr(rank_prefix_matrix, 1, 16) ||
        !ok_ptr(channel_prefix_matrix, 1, 16) || !ok_ptr(recv_channel_prefix_matrix, 1, 16) ||
        !ok_ptr(num_recv_tokens, 1, 16) || !ok_ptr(num_recv_tokens_per_expert, 1, 16) ||
        !ok_ptr(recv_expert_offset, 1, 16) || !ok_ptr(send_head, S * s.P, 16) ||
        !ok_ptr(part_row_base, 1, 16) || !ok_ptr(scratch, 1, 256))
        return MOE_ERR_INVALID_ARG;
    if (scratch_bytes < moe_scratch_bytes(shape)) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_notify(s, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                                   rank_prefix_matrix, channel_prefix_matrix,
                                   recv_channel_prefix_matrix, num_recv_tokens,
                                   num_recv_tokens_per_expert, recv_expert_offset, send_head,
                                   part_row_base, scratch, static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* topk_idx,
                        const float* topk_weights, const int32_t* send_head,
                        const int64_t* part_row_base, void* recv_arena, int64_t arena_rows,
                        int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                        int32_t* err, void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if (arena_rows < 0) return MOE_ERR_INVALID_ARG;
    if (!ok_ptr(x, S * s.H, 16) || !ok_ptr(topk_idx, S * s.K, 16) || !ok_ptr(send_head, S * s.P, 16) ||
        !ok_ptr(part_row_base, 1, 16) || !ok_ptr(recv_arena, arena_rows, 16) ||
        !ok_opt(recv_src_idx, 16) || !ok_opt(recv_topk_idx, 16) || !ok_opt(recv_topk_weights, 16) ||
        !ok_opt(topk_weights, 16) || !ok_opt(err, 4))
        return MOE_ERR_INVALID_ARG;
    if (recv_topk_weights && !topk_weights && S > 0) return MOE_ERR_INVALID_ARG;
    DispatchArgs a{};
    a.P = s.P;
    a.E = s.E;
    a.K = s.K;
    a.H = s.H;
    a.epr = s.E / s.P;
    a.S = S;
    a.T = S / s.P;
    a.x = x;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.send_head = send_head;
    a.part_row_base = part_row_base;
    a.arena = static_cast<uint8_t*>(recv_arena);
    a.arena_rows = arena_rows;
    a.stride = moe_slot_stride(s.H, s.quant);
    a.scale_off = round_up(static_cast<int64_t>(s.H) * (s.quant ? 1 : 2), 32);
    a.triple_off = a.scale_off + 32;
    a.recv_src_idx = recv_src_idx;
    a.recv_topk_idx = recv_topk_idx;
    a.recv_topk_weights = recv_topk_weights;
    a.err = err;
    a.row_bytes = static_cast<uint32_t>(s.H) * 2u;
    return from_cuda(launch_dispatch(s, a, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const moe_shape* shape, const void* y, int64_t y_row_stride,
                       const int64_t* part_row_base, int64_t arena_rows, const int32_t* send_head,
                       const int32_t* topk_idx, const float* topk_weights, uint16_t* out, int32_t* err,
                       void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if (arena_rows < 0 || y_row_stride < 2 * static_cast<int64_t>(s.H) || y_row_stride % 16 != 0)
        return MOE_ERR_INVALID_ARG;
    if (!ok_ptr(y, arena_rows, 16) || !ok_ptr(part_row_base, 1, 16) || !ok_ptr(send_head, S * s.P, 16) ||
        !ok_ptr(topk_idx, S * s.K, 16) || !ok_opt(topk_weights, 16) || !ok_ptr(out, S * s.H, 16) ||
        !ok_opt(err, 4))
        return MOE_ERR_INVALID_ARG;
    CombineArgs a{};
    a.P = s.P;
    a.E = s.E;
    a.K = s.K;
    a.H = s.H;
    a.epr = s.E / s.P;
    a.S = S;
    a.y = static_cast<const uint8_t*>(y);
    a.y_stride = y_row_stride;
    a.part_row_base = part_row_base;
    a.arena_rows = arena_rows;
    a.send_head = send_head;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.out = out;
    a.err = err;
    return from_cuda(launch_combine(s, a, static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_fused(const moe_shape* shape, const uint16_t* x, const int32_t* topk_idx,
                              const float* topk_weights, int32_t* num_tokens_per_rank,
                              int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                              uint32_t* is_token_in_rank_bits, int32_t* rank_prefix_matrix,
                              int32_t* channel_prefix_matrix, int32_t* recv_channel_prefix_matrix,
                              int32_t* num_recv_tokens, int32_t* num_recv_tokens_per_expert,
                              int32_t* recv_expert_offset, int32_t* send_head, int64_t* part_row_base,
                              void* recv_arena, int64_t arena_rows, int32_t* recv_src_idx,
                              int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* err, void* scratch,
                              int64_t scratch_bytes, void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (!fused_supported(s)) return MOE_ERR_UNSUPPORTED;
    const int64_t S = s.S;
    if (arena_rows < 0) return MOE_ERR_INVALID_ARG;
    if (!ok_ptr(x, S * s.H, 16) || !ok_ptr(topk_idx, S * s.K, 16) || !ok_opt(topk_weights, 16) ||
        !ok_ptr(num_tokens_per_rank, 1, 16) || !ok_ptr(num_tokens_per_expert, 1, 16) ||
        !ok_ptr(is_token_in_rank, S * s.P, 16) || !ok_opt(is_token_in_rank_bits, 16) ||
        !ok_ptr(rank_prefix_matrix, 1, 16) || !ok_ptr(channel_prefix_matrix, 1, 16) ||
        !ok_ptr(recv_channel_prefix_matrix, 1, 16) || !ok_ptr(num_recv_tokens, 1, 16) ||
        !ok_ptr(num_recv_tokens_per_expert, 1, 16) || !ok_ptr(recv_expert_offset, 1, 16) ||
        !ok_ptr(send_head, S * s.P, 16) || !ok_ptr(part_row_base, 1, 16) || !ok_ptr(recv_arena, arena_rows, 16) ||
        !ok_opt(recv_src_idx, 16) || !ok_opt(recv_topk_idx, 16) || !ok_opt(recv_topk_weights, 16) ||
        !ok_opt(err, 4) || !ok_ptr(scratch, 1, 256))
        return MOE_ERR_INVALID_ARG;
    if (recv_topk_weights && !topk_weights && S > 0) return MOE_ERR_INVALID_ARG;
    if (scratch_bytes < moe_scratch_bytes(shape)) return MOE_ERR_INVALID_ARG;
    DispatchArgs a{};
    a.P = s.P;
    a.E = s.E;
    a.K = s.K;
    a.H = s.H;
    a.epr = s.E / s.P;
    a.S = S;
    a.T = S / s.P;
    a.x = x;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.send_head = send_head;
    a.part_row_base = part_row_base;
    a.arena = static_cast<uint8_t*>(recv_arena);
    a.arena_rows = arena_rows;
    a.stride = moe_slot_stride(s.H, 0);
    a.scale_off = round_up(static_cast<int64_t>(s.H) * 2, 32);
    a.triple_off = a.scale_off + 32;
    a.recv_src_idx = recv_src_idx;
    a.recv_topk_idx = recv_topk_idx;
    a.recv_topk_weights = recv_topk_weights;
    a.err = err;
    a.row_bytes = static_cast<uint32_t>(s.H) * 2u;
    return from_cuda(launch_fused(s, x, topk_idx, topk_weights, num_tokens_per_rank, num_tokens_per_expert,
                                  is_token_in_rank, is_token_in_rank_bits, rank_prefix_matrix,
                                  channel_prefix_matrix, recv_channel_prefix_matrix, num_recv_tokens,
                                  num_recv_tokens_per_expert, recv_expert_offset, send_head, part_row_base, a,
                                  err, scratch, static_cast<cudaStream_t>(stream)));
}

moe_status moe_notify_expert(const moe_shape* shape, const int32_t* topk_idx,
                             const int32_t* num_recv_tokens_per_expert, const int32_t* recv_expert_offset,
                             int32_t* slot_row, int64_t* expert_part_base, void* scratch,
                             int64_t scratch_bytes, void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if (!ok_ptr(topk_idx, S * s.K, 16) || !ok_ptr(num_recv_tokens_per_expert, 1, 16) ||
        !ok_ptr(recv_expert_offset, 1, 16) || !ok_ptr(slot_row, S * s.K, 16) ||
        !ok_ptr(expert_part_base, 1, 16) || !ok_ptr(scratch, 1, 256))
        return MOE_ERR_INVALID_ARG;
    if (scratch_bytes < moe_scratch_bytes(shape)) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_notify_expert(s, topk_idx, num_recv_tokens_per_expert, recv_expert_offset,
                                          slot_row, expert_part_base, scratch,
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_expert(const moe_shape* shape, const uint16_t* x, const int32_t* topk_idx,
                               const float* topk_weights, const int32_t* slot_row,
                               const int64_t* expert_part_base, void* recv_arena, int64_t arena_rows,
                               int32_t* recv_src_idx, float* recv_weight, int32_t* err, void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if (arena_rows < 0) return MOE_ERR_INVALID_ARG;
    if (!ok_ptr(x, S * s.H, 16) || !ok_ptr(topk_idx, S * s.K, 16) || !ok_ptr(slot_row, S * s.K, 16) ||
        !ok_ptr(expert_part_base, 1, 16) || !ok_ptr(recv_arena, arena_rows, 16) ||
        !ok_opt(recv_src_idx, 16) || !ok_opt(recv_weight, 16) || !ok_opt(topk_weights, 16) ||
        !ok_opt(err, 4))
        return MOE_ERR_INVALID_ARG;
    DispatchArgs a{};
    a.P = s.P;
    a.E = s.E;
    a.K = s.K;
    a.H = s.H;
    a.epr = s.E / s.P;
    a.S = S;
    a.T = S / s.P;
    a.x = x;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.part_row_base = expert_part_base;
    a.arena = static_cast<uint8_t*>(recv_arena);
    a.arena_rows = arena_rows;
    a.stride = moe_slot_stride(s.H, s.quant);
    a.scale_off = round_up(static_cast<int64_t>(s.H) * (s.quant ? 1 : 2), 32);
    a.triple_off = a.scale_off + 32;
    a.recv_src_idx = recv_src_idx;
    a.err = err;
    a.row_bytes = static_cast<uint32_t>(s.H) * 2u;
    a.slot_row = slot_row;
    a.recv_weight = recv_weight;
    return from_cuda(launch_dispatch_expert(s, a, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_expert(const moe_shape* shape, const void* y, int64_t y_row_stride,
                              const int64_t* expert_part_base, int64_t arena_rows, const int32_t* slot_row,
                              const int32_t* topk_idx, const float* topk_weights, uint16_t* out,
                              int32_t* err, void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if (arena_rows < 0 || y_row_stride < 2 * static_cast<int64_t>(s.H) || y_row_stride % 16 != 0)
        return MOE_ERR_INVALID_ARG;
    if (!ok_ptr(y, arena_rows, 16) || !ok_ptr(expert_part_base, 1, 16) || !ok_ptr(slot_row, S * s.K, 16) ||
        !ok_ptr(topk_idx, S * s.K, 16) || !ok_opt(topk_weights, 16) || !ok_ptr(out, S * s.H, 16) ||
        !ok_opt(err, 4))
        return MOE_ERR_INVALID_ARG;
    CombineArgs a{};
    a.P = s.P;
    a.E = s.E;
    a.K = s.K;
    a.H = s.H;
    a.epr = s.E / s.P;
    a.S = S;
    a.y = static_cast<const uint8_t*>(y);
    a.y_stride = y_row_stride;
    a.part_row_base = expert_part_base;
    a.arena_rows = arena_rows;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.out = out;
    a.err = err;
    a.slot_row = slot_row;
    return from_cuda(launch_combine_expert(s, a, static_cast<cudaStream_t>(stream)));
}

#ifdef MOE_PROFILE
moe_status moe_profile_attach(void* slots, int64_t bytes) {
    const int64_t need = static_cast<int64_t>(kProfKernels) * kProfCtas * kProfPhases * 8;
    if (slots != nullptr && (bytes < need || !aligned(slots, 16))) return MOE_ERR_INVALID_ARG;
    cudaError_t (*attach[])(void*) = {prof_attach_layout, prof_attach_notify, prof_attach_dispatch,
                                      prof_attach_combine, prof_attach_fused, prof_attach_expert};
    for (auto f : attach)
        if (f(slots) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}
#endif

moe_status moe_test_fused_barrier(uint32_t spin_limit, int32_t skip_cta) {
    if (spin_limit == 0) return MOE_ERR_INVALID_ARG;
    arm_fused_barrier_test(spin_limit, skip_cta);
    return MOE_OK;
}

moe_status moe_pad_partitions(const moe_shape* shape, const int32_t* num_recv_tokens,
                              const int64_t* part_row_base, void* recv_arena, int64_t arena_rows,
                              int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                              void* stream) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    if (arena_rows < 0) return MOE_ERR_INVALID_ARG;
    if (!ok_ptr(num_recv_tokens, 1, 16) || !ok_ptr(part_row_base, 1, 16) ||
        !ok_ptr(recv_arena, arena_rows, 16) || !ok_opt(recv_src_idx, 16) || !ok_opt(recv_topk_idx, 16) ||
        !ok_opt(recv_topk_weights, 16))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_pad(*shape, num_recv_tokens, part_row_base, static_cast<uint8_t*>(recv_arena),
                                arena_rows, recv_src_idx, recv_topk_idx, recv_topk_weights,
                                static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
