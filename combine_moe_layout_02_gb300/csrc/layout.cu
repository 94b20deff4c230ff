// layout.cu -- routing tables from topk_idx (moe_layout).
//
// Computes, per source rank s, num_tokens_per_rank[s][d], num_tokens_per_expert[s][e]
// and the token -> rank table is_token_in_rank[g][d] (plus its packed form), as
// described in "Ascend DeepEP MoE Dispatch Optimization", sections
// "从 Python 接口进入真实调用链" and "Dispatch handle 六项分别保存什么"; the
// destination rank of an expert is expert_id / experts_per_rank (section
// "一条 token 如何走完 MoE").
//
// Design (sm_103a): one thread-block cluster per source rank, its CTAs taking
// consecutive token ranges of that rank, one thread per token.
//  * Expert histogram: one shared-memory histogram per block, one integer
//    atomic add per (token, k) slot; the counts do not depend on the order of
//    the adds. (Compiled with -DMOE_LAYOUT_MATCH_HIST, the histograms are
//    atomics-free instead: each warp keeps its own sub-histogram, groups its
//    lanes by key with __match_any_sync and lets the lowest lane of a group
//    add the group's size; the sub-histograms are summed in warp order. Same
//    results; the atomic form measured faster on GB300.)
//  * A token's destination ranks are a bit mask (in registers up to 128
//    ranks); the rank of expert e is e / (E/P) by a multiply-shift. Rank
//    counts: up to 32 ranks, one __ballot_sync + __popc per rank over the
//    warp's tokens; above that, a histogram (the same form as the expert
//    one) of each token's first slot on each rank.
//  * The block's slice of is_token_in_rank is written from the packed-bit
//    tile with 16-byte stores: the slice of rows [g0, g0+n) is one contiguous
//    span, each 16-byte chunk made from 16 bits.
//  * The CTAs of the cluster then add their block totals through distributed
//    shared memory, in CTA order, each CTA writing a share of the source
//    rank's num_tokens_per_rank / num_tokens_per_expert row. No second pass
//    over global memory and no cross-cluster synchronisation.
//  * A source rank held by one CTA (T <= 512 tokens) skips the cluster
//    exchange: its totals go straight from shared memory.
//  * A one-block tail kernel folds the clusters' out-of-range flags into the
//    caller's error word (only when an error word is given). It lets the next
//    kernel be scheduled at once, then waits for layout_kernel. (The fold can
//    be done inside layout_kernel, by the last source rank to finish, with a
//    counter in scratch; measured on GB300, the next kernel, moe_notify's,
//    then runs up to twice as slowly when its grid waits on layout_kernel's
//    directly, which costs more than this launch at every size measured.)
#include "moe_device.cuh"

namespace moe {
namespace {

#ifdef MOE_LAYOUT_MATCH_HIST
constexpr bool kAtomicHist = false;
#else
constexpr bool kAtomicHist = true;
#endif

constexpr int kLayoutThreads = 512;         // block size limit: one CTA holds up to 512 tokens
constexpr int kLayoutClusterThreads = 256;  // block size of the CTAs of a cluster
constexpr int kLayoutMaxCluster = 16;
constexpr size_t kLayoutSmemBudget = 96 * 1024;

struct LayoutSmem {
    size_t off_rank, off_tot, off_gat, off_bits, total;
};

// hist [E] (atomic) or [warps][E]; rank counts [warps][P]; block totals
// [P + E + 1]; the peers' totals of this CTA's columns [P + E + 1 + 16];
// packed-bit tile [tb][W].
__host__ __device__ inline LayoutSmem layout_smem(int P, int E, int tb) {
    const int nwarps = tb / 32;
    const int W = (P + 31) / 32;
    const int64_t hist = kAtomicHist ? E : static_cast<int64_t>(nwarps) * E;
    LayoutSmem l;
    l.off_rank = static_cast<size_t>(hist) * 4;
    l.off_tot = l.off_rank + static_cast<size_t>(nwarps) * P * 4;
    l.off_gat = static_cast<size_t>(round_up(static_cast<int64_t>(l.off_tot) + (P + E + 1) * 4, 16));
    l.off_bits = static_cast<size_t>(round_up(static_cast<int64_t>(l.off_gat) + (P + E + 1 + 16) * 4, 16));
    l.total = l.off_bits + static_cast<size_t>(tb) * W * 4;
    return l;
}

// Add 1 to h[key] for every lane with `valid`. The grouped form: lanes with
// the same key form one group (__match_any_sync) and its lowest lane adds the
// group's size, so h is private to the warp and no two lanes of one
// instruction touch the same counter. The atomic form adds per lane. Every
// lane of the warp must call this (the grouped form is a warp collective).
__device__ __forceinline__ void hist_add(int32_t* h, int key, bool valid, int lane) {
    if (kAtomicHist) {
        if (valid) atomicAdd(h + key, 1);
    } else {
        const uint32_t grp = __match_any_sync(0xffffffffu, valid ? key : -1 - lane);
        if (valid && (__ffs(grp) - 1) == lane) h[key] += __popc(grp);
    }
}

// Four bits (bit i -> byte i) as four 0/1 bytes.
__device__ __forceinline__ uint32_t expand4(uint32_t nib) { return (nib * 0x00204081u) & 0x01010101u; }

// Write the is_token_in_rank bytes of n tokens, [n][P] from the packed-bit
// tile [n][W], to dst (one contiguous span). 16 bytes per store where the
// span is 16-byte aligned; each 16-byte chunk is made from 16 bits of the
// tile (bit i -> byte i).
__device__ inline void write_itr_span(uint8_t* dst, const uint32_t* tile, int n, int P, int W, int tid,
                                      int nthreads) {
    const int nbytes = n * P;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0 && ((P & 15) == 0 || (16 % P) == 0)) {
        const int nv = nbytes >> 4;
        for (int i = tid; i < nv; i += nthreads) {
            uint32_t m;
            if ((P & 15) == 0) {
                const int t = (i << 4) / P;
                const int d0 = (i << 4) - t * P;
                m = (tile[t * W + (d0 >> 5)] >> (d0 & 31)) & 0xffffu;
            } else {  // P in {1, 2, 4, 8}: 16 / P tokens per chunk, one word each
                const int per = 16 / P;
                m = 0u;
                for (int j = 0; j < per; ++j) m |= (tile[i * per + j] & ((1u << P) - 1u)) << (j * P);
            }
            reinterpret_cast<uint4*>(dst)[i] =
                make_uint4(expand4(m & 15u), expand4((m >> 4) & 15u), expand4((m >> 8) & 15u), expand4(m >> 12));
        }
        done = nv << 4;
    }
    for (int b = done + tid; b < nbytes; b += nthreads) {
        const int t = b / P;
        const int d = b - t * P;
        dst[b] = static_cast<uint8_t>((tile[t * W + (d >> 5)] >> (d & 31)) & 1u);
    }
}

// Grid: P clusters of cs CTAs; cluster s handles source rank s, CTA r of it
// the r-th block of the balanced split of the rank's T tokens. WR is the
// number of 32-rank mask words a thread keeps in registers: 1 (P <= 32),
// 4 (P <= 128) or 0 (the mask lives in the shared tile). epr_magic =
// ceil(2^32 / (E / P)): the rank of expert e (< 2^12) is (e * epr_magic) >> 32.
// Shape constants of a launch, split on the host so that the kernel does no
// integer division: T tokens per source rank, cs CTAs per cluster, CTA r
// taking the r-th block of the balanced split of T over cs (tq, tr).
struct LayoutParams {
    int32_t P, E, K, T, cs, tq, tr;
    uint64_t epr_magic;
    const int32_t* topk_idx;
    uint8_t* itr;
    uint32_t* bits;
    int32_t *ntpr, *ntpe, *bad_flags;
};

template <int WR>
__global__ void __launch_bounds__(kLayoutThreads) layout_kernel(const LayoutParams a) {
    pdl_wait_then_release();
    const int32_t P = a.P, E = a.E, K = a.K;
    const int64_t T = a.T;
    const uint64_t epr_magic = a.epr_magic;
    const int32_t* __restrict__ topk_idx = a.topk_idx;
    uint8_t* __restrict__ itr = a.itr;
    uint32_t* __restrict__ bits = a.bits;
    int32_t* __restrict__ ntpr = a.ntpr;
    int32_t* __restrict__ ntpe = a.ntpe;
    int32_t* __restrict__ bad_flags = a.bad_flags;
    extern __shared__ __align__(16) unsigned char smem[];
    const int tb = blockDim.x;
    const int nwarps = tb >> 5;
    const int W = (P + 31) >> 5;
    const LayoutSmem L = layout_smem(P, E, tb);
    int32_t* hist = reinterpret_cast<int32_t*>(smem);                      // see layout_smem
    int32_t* rcnt = reinterpret_cast<int32_t*>(smem + L.off_rank);         // [nwarps][P]
    int32_t* tot = reinterpret_cast<int32_t*>(smem + L.off_tot);           // [P + E + 1]
    int32_t* gat = reinterpret_cast<int32_t*>(smem + L.off_gat);           // [cs][span]
    uint32_t* tile_bits = reinterpret_cast<uint32_t*>(smem + L.off_bits);  // [tb][W]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cs = a.cs;
    const int r = static_cast<int>(cluster_ctarank());
    const int64_t s = cluster_id_x();
    const int64_t tbeg = static_cast<int64_t>(r) * a.tq + min(r, a.tr);
    const int64_t tend = tbeg + a.tq + (r < a.tr ? 1 : 0);

    MOE_PROF_BEGIN(kProfLayout);
    for (int i = tid; i < static_cast<int>(L.off_tot / 4); i += tb) reinterpret_cast<int32_t*>(smem)[i] = 0;
    __syncthreads();

    int bad = 0;
    int32_t* my_hist = kAtomicHist ? hist : hist + warp * E;
    int32_t* my_rcnt = rcnt + warp * P;
    uint32_t* my_bits = tile_bits + tid * W;
    const bool vec = (K & 3) == 0;
    // The last chunk's rows are written after the cluster exchange: a cluster
    // barrier's release would otherwise wait for those stores to complete.
    int64_t last_g0 = 0;
    int last_n = 0;
    for (int64_t t0 = tbeg; t0 < tend; t0 += tb) {
        const int n = static_cast<int>(min(static_cast<int64_t>(tb), tend - t0));
        const int64_t g0 = s * T + t0;
        const bool active = tid < n;
        const int64_t g = g0 + tid;
        uint32_t m[WR > 0 ? WR : 1];
#pragma unroll
        for (int w = 0; w < (WR > 0 ? WR : 1); ++w) m[w] = 0u;
        if (WR == 0)
            for (int w = 0; w < W; ++w) my_bits[w] = 0u;
        // One (token, k) slot: expert histogram, rank mask, first-of-rank count.
        auto slot = [&](int32_t e) {
            const bool valid = e >= 0 && e < E;
            if (e >= E) bad = 1;
            hist_add(my_hist, e, valid, lane);
            const int d = valid ? static_cast<int>((static_cast<uint64_t>(e) * epr_magic) >> 32) : 0;
            const uint32_t bit = 1u << (d & 31);
            bool first;
            if (WR == 1) {
                first = valid && !(m[0] & bit);
                if (valid) m[0] |= bit;
            } else if (WR > 1) {
                // Word d >> 5 of the mask, selected without indexing
                // (an indexed register array would live in local memory).
                const uint32_t hi = static_cast<uint32_t>(d >> 5);
                const uint32_t b0 = (valid && hi == 0u) ? bit : 0u, b1 = (valid && hi == 1u) ? bit : 0u;
                const uint32_t b2 = (valid && hi == 2u) ? bit : 0u, b3 = (valid && hi == 3u) ? bit : 0u;
                first = valid && !((m[0] & b0) | (m[WR > 1 ? 1 : 0] & b1) | (m[WR > 2 ? 2 : 0] & b2) |
                                   (m[WR > 3 ? 3 : 0] & b3));
                m[0] |= b0;
                if (WR > 1) m[WR > 1 ? 1 : 0] |= b1;
                if (WR > 2) m[WR > 2 ? 2 : 0] |= b2;
                if (WR > 3) m[WR > 3 ? 3 : 0] |= b3;
            } else {
                const uint32_t cur = valid ? my_bits[d >> 5] : 0u;
                first = valid && !(cur & bit);
                if (first) my_bits[d >> 5] = cur | bit;
            }
            if (WR != 1) hist_add(my_rcnt, d, first, lane);
        };
        if (vec) {
#pragma unroll 2
            for (int k4 = 0; k4 < K; k4 += 4) {
                const int4 v = active ? __ldg(reinterpret_cast<const int4*>(topk_idx + g * K + k4))
                                      : make_int4(-1, -1, -1, -1);
                slot(v.x);
                slot(v.y);
                slot(v.z);
                slot(v.w);
            }
        } else {
#pragma unroll 4
            for (int k = 0; k < K; ++k) slot(active ? __ldg(topk_idx + g * K + k) : -1);
        }
        if (WR > 0) {
#pragma unroll
            for (int w = 0; w < (WR > 0 ? WR : 1); ++w)
                if (w < W) my_bits[w] = m[w];  // W <= WR: constant indices after unrolling
        }
        if (WR == 1) {
            // Tokens of this warp per rank, 4 ranks per warp reduction: each
            // lane's 4 rank bits as 4 bytes (counts <= 32 fit a byte).
            for (int d4 = 0; d4 < P; d4 += 4) {
                const uint32_t c4 = __reduce_add_sync(0xffffffffu, expand4((m[0] >> d4) & 15u));
                if (lane < 4 && d4 + lane < P) my_rcnt[d4 + lane] += static_cast<int32_t>((c4 >> (8 * lane)) & 0xffu);
            }
        }
        MOE_STAMP(1);
        __syncthreads();
        MOE_STAMP(2);
        if (t0 + tb < tend) {  // an earlier chunk: written now, its tile is reused
            write_itr_span(itr + g0 * P, tile_bits, n, P, W, tid, tb);
            if (bits) {
                uint32_t* dst = bits + g0 * W;
                for (int i = tid; i < n * W; i += tb) dst[i] = tile_bits[i];
            }
            __syncthreads();
        } else {
            last_g0 = g0;
            last_n = n;
        }
    }

    // Block totals, summed over warps in warp order.
    for (int j = tid; j < P; j += tb) {
        int32_t sum = 0;
#pragma unroll 8
        for (int w = 0; w < nwarps; ++w) sum += rcnt[w * P + j];
        tot[j] = sum;
    }
    MOE_STAMP(8);
    for (int j = tid; j < E; j += tb) {
        int32_t sum = 0;
        if (kAtomicHist) {
            sum = hist[j];
        } else {
            for (int w = 0; w < nwarps; ++w) sum += hist[w * E + j];
        }
        tot[P + j] = sum;
    }
    MOE_STAMP(9);
    const int any_bad = __syncthreads_or(bad);
    MOE_STAMP(10);
    if (tid == 0) tot[P + E] = any_bad;
    MOE_STAMP(3);

    if (cs == 1) {  // the CTA holds the whole source rank: no cluster exchange
        if (last_n > 0) {
            write_itr_span(itr + last_g0 * P, tile_bits, last_n, P, W, tid, tb);
            if (bits) {
                uint32_t* dst = bits + last_g0 * W;
                for (int i = tid; i < last_n * W; i += tb) dst[i] = tile_bits[i];
            }
        }
        MOE_STAMP(4);  // phases 4 and 5 (the cluster exchange) end here
        MOE_STAMP(5);
        for (int j = tid; j < P + E; j += tb) {
            if (j < P)
                ntpr[s * P + j] = tot[j];
            else
                ntpe[s * E + (j - P)] = tot[j];
        }
        if (tid == 0 && bad_flags) bad_flags[s] = any_bad != 0;
        MOE_STAMP(6);
        MOE_STAMP(7);
        MOE_PROF_END();
        return;
    }
    // Cluster reduction: CTA r sums columns [r*span, (r+1)*span) over the
    // cluster's CTAs in CTA order. Each (column, peer) pair is read by its
    // own thread, then summed from shared memory.
    cluster_sync_all();
    MOE_STAMP(4);
    const int ncol = P + E + 1;
    const int span = (ncol + cs - 1) / cs;
    const int c0 = min(ncol, r * span), w = min(ncol, c0 + span) - c0;
    for (int i = tid; i < cs * w; i += tb) {
        const int q = i / w, j = i - q * w;
        gat[i] = ld_cluster_s32(cluster_map(tot + c0 + j, q));
    }
    MOE_STAMP(11);
    cluster_arrive();  // done reading the peers; they may exit once all have arrived
    MOE_STAMP(12);
    if (last_n > 0) {
        write_itr_span(itr + last_g0 * P, tile_bits, last_n, P, W, tid, tb);
        if (bits) {
            uint32_t* dst = bits + last_g0 * W;
            for (int i = tid; i < last_n * W; i += tb) dst[i] = tile_bits[i];
        }
    }
    MOE_STAMP(13);
    __syncthreads();
    MOE_STAMP(5);
    for (int j = tid; j < w; j += tb) {
        int32_t sum = 0;
#pragma unroll 4
        for (int q = 0; q < cs; ++q) sum += gat[q * w + j];
        const int col = c0 + j;
        if (col < P)
            ntpr[s * P + col] = sum;
        else if (col < P + E)
            ntpe[s * E + (col - P)] = sum;
        else if (bad_flags)
            bad_flags[s] = sum != 0;
    }
    MOE_STAMP(6);
    // Keep this CTA's totals alive until every peer has read them.
    cluster_wait();
    MOE_STAMP(7);
    MOE_PROF_END();
}

// Fold the per-source out-of-range flags into the caller's error word. It
// lets the next kernel be scheduled before it waits for layout_kernel, so that
// launch overlaps layout_kernel rather than following it; the next kernel
// still waits for this grid to complete before it touches global memory.
__global__ void __launch_bounds__(256)
layout_err_kernel(int32_t P, const int32_t* __restrict__ bad_flags, int32_t* __restrict__ err) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int bad = 0;
    for (int i = threadIdx.x; i < P; i += blockDim.x) bad |= bad_flags[i];
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) *err = bad ? MOE_ERR_TOPK_OUT_OF_RANGE : MOE_OK;
}

// CTAs per source rank (before the residency check of the cluster size) and
// threads per CTA for a shape.
// A source rank of up to kLayoutThreads tokens is one CTA (no cluster
// exchange); a longer one is a cluster of CTAs of about
// kLayoutClusterThreads tokens each. (Measured on GB300, layout + notify
// inside a step: p128_e256_t512 30.0-32.0 us with one 512-thread CTA per
// source rank against 33.2-33.4 us with two of 256; p8_e256_t4096 best with
// 16 CTAs of 256, 13.8-15.1 us, against 8 of 512, 14.5-15.1 us.)
void layout_geometry(const moe_shape& s, int* cs, int* threads) {
    const int64_t T = s.S / s.P;
    int c = 1;  // a power of two
    if (T > kLayoutThreads)
        while (c < kLayoutMaxCluster && static_cast<int64_t>(c) * kLayoutClusterThreads < T) c <<= 1;
    const int64_t n = ceil_div(T, c);
    int tb = static_cast<int>(round_up(n < 32 ? 32 : n, 32));
    if (tb > kLayoutThreads) tb = kLayoutThreads;
    while (tb > 32 && layout_smem(s.P, s.E, tb).total > kLayoutSmemBudget) tb -= 32;
    *cs = c;
    *threads = tb;
}

const void* layout_fn(int P) {
    if (P <= 32) return reinterpret_cast<const void*>(layout_kernel<1>);
    if (P <= 128) return reinterpret_cast<const void*>(layout_kernel<4>);
    return reinterpret_cast<const void*>(layout_kernel<0>);
}

}  // namespace

MOE_PROFILE_UNIT(layout)

LayoutPlan layout_plan(const moe_shape& s) {
    LayoutPlan p;
    layout_geometry(s, &p.cluster, &p.threads);
    p.smem = layout_smem(s.P, s.E, p.threads).total;
    p.scratch_bytes = round_up(static_cast<int64_t>(s.P) * 4, 256);
    return p;
}

cudaError_t launch_layout(const moe_shape& s, const int32_t* topk_idx, int32_t* ntpr, int32_t* ntpe,
                          uint8_t* itr, uint32_t* bits, int32_t* err, void* scratch,
                          cudaStream_t stream) {
    const LayoutPlan p = layout_plan(s);
    int32_t* flags = err ? static_cast<int32_t*>(scratch) : nullptr;
    const void* fn = layout_fn(s.P);
    cudaError_t e = prepare_kernel(fn, p.smem, p.threads, nullptr);
    if (e != cudaSuccess) return e;
    const int cs = cluster_size_for(fn, p.cluster, p.threads, p.smem);
    if (cs < 1) return cudaErrorInvalidConfiguration;
    const int epr = s.E / s.P;
    LayoutParams a{};
    a.P = s.P;
    a.E = s.E;
    a.K = s.K;
    a.T = static_cast<int32_t>(s.S / s.P);
    a.cs = cs;
    a.tq = a.T / cs;
    a.tr = a.T % cs;
    a.epr_magic = ((uint64_t{1} << 32) + static_cast<uint64_t>(epr) - 1) / static_cast<uint64_t>(epr);
    a.topk_idx = topk_idx;
    a.itr = itr;
    a.bits = bits;
    a.ntpr = ntpr;
    a.ntpe = ntpe;
    a.bad_flags = flags;
    const unsigned grid = static_cast<unsigned>(s.P) * cs;
    if (s.P <= 32)
        e = launch_pdl_cluster(layout_kernel<1>, grid, p.threads, p.smem, cs, stream, a);
    else if (s.P <= 128)
        e = launch_pdl_cluster(layout_kernel<4>, grid, p.threads, p.smem, cs, stream, a);
    else
        e = launch_pdl_cluster(layout_kernel<0>, grid, p.threads, p.smem, cs, stream, a);
    if (e != cudaSuccess || !err) return e;
    return launch_pdl(layout_err_kernel, 1u, 256u, 0, stream, s.P, static_cast<const int32_t*>(flags), err);
}

}  // namespace moe
