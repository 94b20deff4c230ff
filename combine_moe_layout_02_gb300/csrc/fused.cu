// fused.cu -- layout + notify + dispatch in one launch (moe_dispatch_fused).
//
// The small-message regime ("Ascend DeepEP MoE Dispatch Optimization", section
// "128P 为什么会放大问题": with small per-peer messages the fixed control cost
// -- routing scan, counts, prefixes -- dominates the payload) is served by one
// persistent cooperative kernel instead of five launches. This follows the
// single-kernel shape of "DeepEP Warp Specialization 深度分析" (dispatch_impl:
// counting, grid reduction and prefix sums, then the copies), here with
// bounded grid barriers instead of inter-GPU signals. Outputs are exactly
// those of moe_layout, moe_notify and moe_dispatch with packed partitions.
//
// Phase A (one warp per (source rank, channel)): distinct ranks per token from
//   topk_idx; is_token_in_rank rows (+ bits); per-channel rank counts (ballots)
//   and expert counts (__match_any_sync leaders into warp-private shared
//   counters) into scratch.
// grid barrier
// Phase B: every CTA rebuilds, in shared memory, the per-source rank counts
//   and their running sum over sources from the channel counts (a few KB for
//   the supported P); CTA 0 writes num_tokens_per_rank, rank_prefix_matrix,
//   num_recv_tokens and part_row_base. Expert tables are spread over all
//   threads. Then one warp per channel writes channel_prefix_matrix,
//   recv_channel_prefix_matrix and the channel's send_head rows.
// grid barrier
// Phase C (one warp per token, all warps of the grid): each warp bulk-loads
//   its token's row into its shared-memory buffer (mbarrier), its lanes
//   bulk-store it to every destination, and the warp writes the triple and
//   side arrays.
//
// Supported: P <= 64, E <= 1024, H <= 8192; larger shapes use the separate
// calls. The grid barrier counter lives in scratch and is zeroed on the
// stream before the launch.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxP = 64;
constexpr int kMaxE = 1024;
constexpr int kMaxH = 8192;

struct FusedArgs {
    int32_t P, E, K, H, C, A, epr;
    int64_t S, T;
    const uint16_t* x;
    const int32_t* topk_idx;
    const float* topk_weights;
    int32_t* ntpr;
    int32_t* ntpe;
    uint8_t* itr;
    uint32_t* bits;
    int32_t* rpm;
    int32_t* cpm;
    int32_t* rcpm;
    int32_t* nrt;
    int32_t* nrtpe;
    int32_t* reo;
    int32_t* send_head;
    int64_t* part_row_base;
    DispatchArgs d;       // payload stage (part_row_base, send_head as above)
    int32_t* ccount;      // scratch [P*C][P]
    int32_t* ecount;      // scratch [P*C][E]
    unsigned int* barrier;  // scratch, zeroed before launch
    int32_t* err;
};

// Bounded grid barrier over all CTAs of a cooperative launch. Returns false
// (and records MOE_ERR_DEVICE_TIMEOUT) if the other CTAs did not arrive in time.
__device__ bool grid_barrier(unsigned int* counter, unsigned int target, int32_t* err) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        int done = 0;
        for (uint32_t i = 0; i < kSpinLimit; ++i) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            if (v >= target) {
                done = 1;
                break;
            }
            __nanosleep(64);
        }
        if (!done) raise_error(err, MOE_ERR_DEVICE_TIMEOUT);
        ok = done;
    }
    __syncthreads();
    return ok != 0;
}

// ---- phase A: counts and the token -> rank table -------------------------------
__device__ void phase_counts(const FusedArgs& a, unsigned char* smem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* hist_e = reinterpret_cast<int32_t*>(smem) + warp * (a.E + a.P);
    int32_t* hist_r = hist_e + a.E;
    const int64_t chans = static_cast<int64_t>(a.P) * a.C;
    const int64_t total_warps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int W = (a.P + 31) / 32;
    for (int64_t ch = static_cast<int64_t>(blockIdx.x) * kWarps + warp; ch < chans; ch += total_warps) {
        const int64_t s = ch / a.C, c = ch % a.C;
        int64_t b, e;
        split_range(a.T, a.C, c, &b, &e);
        for (int i = lane; i < a.E + a.P; i += 32) hist_e[i] = 0;
        __syncwarp();
        for (int64_t t0 = b; t0 < e; t0 += 32) {
            const int64_t t = t0 + lane;
            const bool active = t < e;
            const int64_t g = s * a.T + t;
            uint64_t mask = 0;
            for (int k = 0; k < a.K; ++k) {
                int32_t ex = active ? __ldg(a.topk_idx + g * a.K + k) : -1;
                if (ex >= a.E) {
                    raise_error(a.err, MOE_ERR_TOPK_OUT_OF_RANGE);
                    ex = -1;
                }
                if (ex < 0) ex = -1;
                const uint32_t grp = __match_any_sync(0xffffffffu, ex);
                if (ex >= 0) {
                    if (lane == __ffs(grp) - 1) hist_e[ex] += __popc(grp);
                    mask |= 1ull << (ex / a.epr);
                }
                __syncwarp();
            }
            if (active) {
                uint8_t* row = a.itr + g * a.P;
                for (int d = 0; d < a.P; ++d) row[d] = static_cast<uint8_t>((mask >> d) & 1ull);
                if (a.bits) {
                    for (int w = 0; w < W; ++w) a.bits[g * W + w] = static_cast<uint32_t>(mask >> (32 * w));
                }
            }
            for (int d = 0; d < a.P; ++d) {
                const uint32_t bal = __ballot_sync(0xffffffffu, (mask >> d) & 1ull);
                if (lane == (d & 31)) hist_r[d] += __popc(bal);
            }
            __syncwarp();
        }
        for (int d = lane; d < a.P; d += 32) a.ccount[ch * a.P + d] = hist_r[d];
        for (int x = lane; x < a.E; x += 32) a.ecount[ch * a.E + x] = hist_e[x];
        __syncwarp();
    }
}

// ---- phase B: tables and send_head -------------------------------------------
__device__ void phase_tables(const FusedArgs& a, unsigned char* smem) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.P, C = a.C, E = a.E;
    int32_t* tot = reinterpret_cast<int32_t*>(smem);  // [P][P] per-source rank counts
    int32_t* run = tot + P * P;                        // [P][P] inclusive over sources
    int64_t* prb = reinterpret_cast<int64_t*>(run + P * P);  // [P+1]
    for (int i = tid; i < P * P; i += kThreads) {
        const int s = i / P, d = i % P;
        int32_t sum = 0;
        for (int c = 0; c < C; ++c) sum += __ldcg(a.ccount + (static_cast<int64_t>(s) * C + c) * P + d);
        tot[i] = sum;
    }
    __syncthreads();
    for (int d = tid; d < P; d += kThreads) {
        int32_t r = 0;
        for (int s = 0; s < P; ++s) {
            r += tot[s * P + d];
            run[s * P + d] = r;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int64_t acc = 0;
        for (int d = 0; d < P; ++d) {
            prb[d] = acc;
            acc += run[(P - 1) * P + d];
        }
        prb[P] = acc;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int i = tid; i < P * P; i += kThreads) {
            a.ntpr[i] = tot[i];
            a.rpm[i] = run[i];
        }
        for (int d = tid; d < P; d += kThreads) a.nrt[d] = run[(P - 1) * P + d];
        for (int d = tid; d <= P; d += kThreads) a.part_row_base[d] = prb[d];
    }
    // Expert tables, spread over the grid: num_tokens_per_expert[s][e].
    const int64_t gthreads = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + tid;
    for (int64_t i = gtid; i < static_cast<int64_t>(P) * E; i += gthreads) {
        const int64_t s = i / E, x = i % E;
        int32_t sum = 0;
        for (int c = 0; c < C; ++c) sum += __ldcg(a.ecount + (s * C + c) * E + x);
        a.ntpe[i] = sum;
    }
    const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    const int64_t total_warps = static_cast<int64_t>(gridDim.x) * kWarps;
    // Channel prefixes and send_head, one warp per channel.
    int32_t* base_all = reinterpret_cast<int32_t*>(prb + P + 1);  // [warps][P]
    int32_t* base = base_all + warp * P;
    const int64_t chans = static_cast<int64_t>(P) * C;
    for (int64_t ch = gwarp; ch < chans; ch += total_warps) {
        const int64_t s = ch / C, c = ch % C;
        int64_t b, e;
        split_range(a.T, C, c, &b, &e);
        for (int d = lane; d < P; d += 32) {
            int32_t pre = 0;
            for (int64_t cc = 0; cc < c; ++cc) pre += __ldcg(a.ccount + (s * C + cc) * P + d);
            const int32_t cnt = __ldcg(a.ccount + ch * P + d);
            const int32_t rank_base = s > 0 ? run[(s - 1) * P + d] : 0;
            a.cpm[(s * P + d) * C + c] = pre + cnt;
            a.rcpm[(static_cast<int64_t>(d) * P + s) * C + c] = rank_base + pre;
            base[d] = rank_base + pre;
        }
        __syncwarp();
        const uint32_t below = lanemask_lt();
        for (int64_t t0 = b; t0 < e; t0 += 32) {
            const int64_t t = t0 + lane;
            const bool active = t < e;
            const int64_t g = s * a.T + t;
            const uint8_t* row = a.itr + g * P;
            for (int d = 0; d < P; ++d) {
                const bool has = active && __ldcg(row + d) != 0;
                const uint32_t bal = __ballot_sync(0xffffffffu, has);
                const int32_t bd = base[d];
                if (active) a.send_head[g * P + d] = has ? bd + __popc(bal & below) : -1;
                __syncwarp();
                if (lane == 0) base[d] = bd + __popc(bal);
                __syncwarp();
            }
        }
    }
}

// ---- phase C: payload ------------------------------------------------------------
__device__ void phase_payload(const FusedArgs& a, unsigned char* smem, const int64_t* prb_sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DispatchArgs& d = a.d;
    const uint32_t RB = static_cast<uint32_t>(a.H) * 2u;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem) + warp;
    unsigned char* buf = smem + 128 + static_cast<size_t>(warp) * RB;
    if (lane == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    __syncwarp();
    const int64_t total_warps = static_cast<int64_t>(gridDim.x) * kWarps;
    // Per rank d (one warp): aligned per-expert receive counts and their
    // offsets, summed over the source ranks of num_tokens_per_expert (phase B).
    for (int64_t dr = static_cast<int64_t>(blockIdx.x) * kWarps + warp; dr < a.P; dr += total_warps) {
        int32_t carry = 0;
        for (int l0 = 0; l0 < a.epr; l0 += 32) {
            const int l = l0 + lane;
            int64_t cnt = 0;
            if (l < a.epr) {
                const int64_t x = dr * a.epr + l;
                for (int s = 0; s < a.P; ++s) cnt += __ldcg(a.ntpe + static_cast<int64_t>(s) * a.E + x);
                cnt = round_up(cnt, a.A);
            }
            int32_t incl = static_cast<int32_t>(cnt);
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (l < a.epr) {
                a.nrtpe[dr * a.epr + l] = static_cast<int32_t>(cnt);
                a.reo[dr * a.epr + l] = carry + incl - static_cast<int32_t>(cnt);
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    uint32_t phase = 0;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kWarps + warp; g < a.S; g += total_warps) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, RB);
            bulk_load(buf, a.x + g * a.H, RB, bar);
        }
        const bool ok = mbar_wait(bar, phase);
        phase ^= 1u;
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) raise_error(a.err, MOE_ERR_DEVICE_TIMEOUT);
            break;
        }
        for (int d0 = 0; d0 < a.P; d0 += 32) {
            const int dd = d0 + lane;
            const int32_t sh = dd < a.P ? __ldcg(a.send_head + g * a.P + dd) : -1;
            if (sh >= 0) {
                const int64_t lo = prb_sm[dd], hi = prb_sm[dd + 1], row = lo + sh;
                if (sh < hi - lo && row >= 0 && row < d.arena_rows)
                    bulk_store(d.arena + row * d.stride, buf, RB);
                else
                    raise_error(a.err, MOE_ERR_CAPACITY);
            }
        }
        bulk_commit();
        // triple and side arrays (reads the send_head row this grid wrote)
        {
            const int K = a.K;
            int32_t idx = -1;
            float w = 0.f;
            if (lane < K) {
                idx = __ldg(a.topk_idx + g * K + lane);
                if (a.topk_weights) w = __ldg(a.topk_weights + g * K + lane);
            }
            const int32_t dk = (idx >= 0 && idx < a.E) ? idx / a.epr : -1;
            const int32_t src_rank = static_cast<int32_t>(g / a.T), src_tok = static_cast<int32_t>(g % a.T);
            for (int d0 = 0; d0 < a.P; d0 += 32) {
                const int dd = d0 + lane;
                const int32_t sh = dd < a.P ? __ldcg(a.send_head + g * a.P + dd) : -1;
                uint32_t todo = __ballot_sync(0xffffffffu, sh >= 0);
                while (todo) {
                    const int j = __ffs(todo) - 1;
                    todo &= todo - 1;
                    const int dj = d0 + j;
                    const int32_t shd = __shfl_sync(0xffffffffu, sh, j);
                    const int64_t lo = prb_sm[dj], hi = prb_sm[dj + 1], row = lo + shd;
                    if (shd >= hi - lo || row < 0 || row >= d.arena_rows) continue;
                    const bool on = dk == dj;
                    const uint32_t kb = __ballot_sync(0xffffffffu, on);
                    if (lane < K) {
                        if (d.recv_topk_idx) d.recv_topk_idx[row * K + lane] = on ? idx % a.epr : -1;
                        if (d.recv_topk_weights) d.recv_topk_weights[row * K + lane] = on ? w : 0.f;
                    }
                    if (lane == 0) {
                        if (d.recv_src_idx) d.recv_src_idx[row] = src_tok;
                        int4* tr = reinterpret_cast<int4*>(d.arena + row * d.stride + d.triple_off);
                        tr[0] = make_int4(src_rank, src_tok, kb ? __ffs(kb) - 1 : -1, 0);
                        tr[1] = make_int4(0, 0, 0, 0);
                    }
                }
            }
        }
        bulk_wait_read<0>();
        __syncwarp();
    }
    bulk_wait<0>();
}

__global__ void __launch_bounds__(kThreads, 1) fused_kernel(const FusedArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const unsigned int n = gridDim.x;
    phase_counts(a, smem);
    if (!grid_barrier(a.barrier, n, a.err)) return;
    phase_tables(a, smem);
    if (!grid_barrier(a.barrier, 2 * n, a.err)) return;
    // part_row_base is still in shared memory from phase B (same CTA).
    const int64_t* prb = reinterpret_cast<const int64_t*>(reinterpret_cast<int32_t*>(smem) + 2 * a.P * a.P);
    // Copy it out of the area phase C reuses for its buffers.
    __shared__ int64_t prb_sm[kMaxP + 1];
    for (int i = threadIdx.x; i <= a.P; i += blockDim.x) prb_sm[i] = prb[i];
    // The shared memory written by phases A and B is reused by bulk copies.
    fence_proxy_async_smem();
    __syncthreads();
    phase_payload(a, smem, prb_sm);
}

size_t fused_smem(const moe_shape& s) {
    const size_t a = static_cast<size_t>(kWarps) * (s.E + s.P) * 4;
    const size_t b = static_cast<size_t>(2 * s.P * s.P) * 4 + static_cast<size_t>(s.P + 1) * 8 +
                     static_cast<size_t>(kWarps) * s.P * 4;
    const size_t c = 128 + static_cast<size_t>(kWarps) * s.H * 2;
    size_t m = a > b ? a : b;
    return m > c ? m : c;
}

}  // namespace

bool fused_supported(const moe_shape& s) {
    return s.P <= kMaxP && s.E <= kMaxE && s.H <= kMaxH && s.quant == 0;
}

int64_t fused_scratch_bytes(const moe_shape& s) {
    const int64_t chans = static_cast<int64_t>(s.P) * s.num_channels;
    return round_up(chans * (s.P + s.E) * 4 + 256, 256);
}

cudaError_t launch_fused(const moe_shape& s, const uint16_t* x, const int32_t* topk_idx, const float* topk_weights,
                         int32_t* ntpr, int32_t* ntpe, uint8_t* itr, uint32_t* bits, int32_t* rpm, int32_t* cpm,
                         int32_t* rcpm, int32_t* nrt, int32_t* nrtpe, int32_t* reo, int32_t* send_head,
                         int64_t* part_row_base, const DispatchArgs& d, int32_t* err, void* scratch,
                         cudaStream_t stream) {
    FusedArgs a{};
    a.P = s.P;
    a.E = s.E;
    a.K = s.K;
    a.H = s.H;
    a.C = s.num_channels;
    a.A = s.expert_alignment;
    a.epr = s.E / s.P;
    a.S = s.S;
    a.T = s.S / s.P;
    a.x = x;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.ntpr = ntpr;
    a.ntpe = ntpe;
    a.itr = itr;
    a.bits = bits;
    a.rpm = rpm;
    a.cpm = cpm;
    a.rcpm = rcpm;
    a.nrt = nrt;
    a.nrtpe = nrtpe;
    a.reo = reo;
    a.send_head = send_head;
    a.part_row_base = part_row_base;
    a.d = d;
    const int64_t chans = static_cast<int64_t>(s.P) * s.num_channels;
    unsigned char* sc = static_cast<unsigned char*>(scratch);
    a.barrier = reinterpret_cast<unsigned int*>(sc);
    a.ccount = reinterpret_cast<int32_t*>(sc + 256);
    a.ecount = a.ccount + chans * s.P;
    a.err = err;
    const size_t smem = fused_smem(s);
    cudaError_t e = cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int grid = device_sm_count();  // one CTA per SM: all resident (cooperative launch)
    e = cudaMemsetAsync(a.barrier, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    if (err) {
        e = cudaMemsetAsync(err, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess) return e;
    }
    void* args[] = {&a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fused_kernel), dim3(grid), dim3(kThreads),
                                       args, smem, stream);
}

}  // namespace moe
