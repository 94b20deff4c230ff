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
// The control phases are laid out so that no warp waits on a chain of
// dependent global loads: every count a later phase needs is written where
// that phase reads it contiguously, and loads are issued in batches.
//
// Start: each warp issues the bulk loads of its first token rows into its
//   own ring of row buffers (x is an input, so the copies need no barrier).
// Phase A (one warp per channel ch = (source rank s, channel c)): for 32
//   tokens at a time (one per lane), the destination-rank mask of each token
//   (topk_idx) and the expert counts (shared-memory integer atomics);
//   is_token_in_rank rows (+ bits); then, lanes over destination ranks, the
//   position of each token among the channel's tokens sent to each rank,
//   written to send_head (local positions, made global in phase C); the
//   channel's rank counts go to ccT[d][ch] (rank-major, so phase B scans a
//   contiguous column) and its expert counts to ecount[ch][e].
// grid barrier
// Phase B (one warp per task): destination rank d scans column ccT[d][.] over
//   the flattened (s, c) order: the exclusive prefix is the channel's first
//   row on d, which is recv_channel_prefix_matrix and the base of send_head
//   ("internode.cu", notify: prefix sums over (source, channel)); the same
//   column gives channel_prefix_matrix, num_tokens_per_rank,
//   rank_prefix_matrix and num_recv_tokens. Expert e sums its channel counts
//   per source (num_tokens_per_expert) and in total (aligned: the receive
//   counts per expert).
// grid barrier
// Phase C: every CTA scans num_recv_tokens into part_row_base (shared
//   memory); one warp per rank scans its experts' aligned counts into
//   recv_expert_offset; then one warp per token stream: send_head entries
//   become global rows (local position + the channel's first row,
//   recv_channel_prefix_matrix[d][s][c]), one lane per destination
//   bulk-stores the row from the ring, the warp writes the triple and side
//   arrays and refills the ring. The routing of the next token is loaded
//   while the current one is copied.
//
// Supported: P <= 64, E <= 1024, H <= 8192, K <= 16, P * num_channels <=
// 4096, bf16; larger shapes use the separate calls. The grid barrier counter
// lives in scratch and is zeroed by a one-thread kernel launched just before
// (both launches use programmatic dependent launch, so the fused kernel is
// scheduled while earlier work drains); err is cleared by the kernel itself.
#include <atomic>

#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxP = 64;
constexpr int kMaxE = 1024;
constexpr int kMaxH = 8192;
constexpr int kMaxPC = 4096;  // P * num_channels (per-warp column in shared memory)
constexpr int kMaxK = 16;
constexpr int kMaxNB = 4;     // row buffers per warp
constexpr int kBarBytes = kWarps * kMaxNB * 8;
constexpr int kSeg = 16;      // column elements per lane per block in phase B
constexpr int kSumUnroll = 16;
// Dynamic shared memory a CTA may use next to the kernel's static shared
// memory (sm_100-class opt-in limit 227 KB, less a margin for static data).
constexpr int kSmemBudget = 227 * 1024 - 1024;
// CTAs per SM tried first; a shape whose row buffers do not fit in that share
// of the SM's shared memory runs one CTA per SM.
#ifndef MOE_FUSED_CTAS_PER_SM
#define MOE_FUSED_CTAS_PER_SM 2
#endif
constexpr int kCtasPerSm = MOE_FUSED_CTAS_PER_SM;

struct FusedArgs {
    int32_t P, E, K, H, C, A, epr, nb;
    uint32_t cq, cr;        // T = cq * C + cr: channels c < cr hold cq + 1 tokens, the rest cq
    int64_t S, T, PC, PCp;
    uint32_t ab_off;        // byte offset of the phase A / B region in dynamic shared memory
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
    DispatchArgs d;         // payload stage (part_row_base, send_head as above)
    int32_t* ccT;           // scratch [P][PCp]: tokens of channel ch sent to rank d
    int32_t* ecount;        // scratch [P*C][E]: slots of channel ch on expert e
    unsigned int* barrier;  // scratch, zeroed before launch
    int32_t* err;
    uint32_t spin_limit;    // polls of a grid barrier before it gives up (kSpinLimit)
    int64_t skip_arrival;   // CTA that leaves out its first arrival (test hook), else -1
};

// Bounded grid barrier over all CTAs of a cooperative launch: at most
// spin_limit polls. Returns false (and records MOE_ERR_DEVICE_TIMEOUT) if the
// other CTAs did not arrive in time. skip_arrival (set only by the test hook
// moe_test_fused_barrier) leaves this CTA's arrival out, so that every CTA's
// wait runs out.
__device__ bool grid_barrier(unsigned int* counter, unsigned int target, int32_t* err, uint32_t spin_limit,
                             bool skip_arrival) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (!skip_arrival) atomicAdd(counter, 1u);
        int done = 0;
        for (uint32_t i = 0; i < spin_limit; ++i) {
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

__device__ __forceinline__ int32_t warp_incl_scan(int32_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// 4 mask bits -> 4 bytes of 0 / 1 (little-endian).
__device__ __forceinline__ uint32_t bytes_of_bits(uint32_t nib) {
    return (nib & 1u) | ((nib & 2u) << 7) | ((nib & 4u) << 14) | ((nib & 8u) << 21);
}

// is_token_in_rank row of one token from its rank mask.
__device__ __forceinline__ void write_itr_row(uint8_t* row, uint64_t mask, int P) {
    if ((P & 15) == 0) {
        for (int q = 0; q < P; q += 16) {
            const uint32_t m16 = static_cast<uint32_t>(mask >> q);
            *reinterpret_cast<uint4*>(row + q) =
                make_uint4(bytes_of_bits(m16 & 15u), bytes_of_bits((m16 >> 4) & 15u),
                           bytes_of_bits((m16 >> 8) & 15u), bytes_of_bits((m16 >> 12) & 15u));
        }
    } else if ((P & 3) == 0) {
        for (int q = 0; q < P; q += 4)
            *reinterpret_cast<uint32_t*>(row + q) = bytes_of_bits(static_cast<uint32_t>(mask >> q) & 15u);
    } else {
        for (int q = 0; q < P; ++q) row[q] = static_cast<uint8_t>((mask >> q) & 1ull);
    }
}

// ---- phase A: masks, local positions, channel counts ------------------------------
// Returns true if this thread saw an expert id >= E.
__device__ bool phase_counts(const FusedArgs& a, int32_t* region) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = a.P, E = a.E, K = a.K;
    int32_t* hist = region + warp * E;
    const int64_t total_warps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int W = (P + 31) / 32;
    bool bad = false;
    // Channels are dealt warp-major (warp w of every CTA before warp w + 1), so
    // a few hundred of them spread over all SMs rather than the first CTAs'.
    for (int64_t ch = static_cast<int64_t>(warp) * gridDim.x + blockIdx.x; ch < a.PC; ch += total_warps) {
        const uint32_t s32 = static_cast<uint32_t>(ch) / static_cast<uint32_t>(a.C);
        const int64_t s = s32, c = ch - static_cast<int64_t>(s32) * a.C;
        int64_t b, e;
        split_range(a.T, a.C, c, &b, &e);
        for (int i = lane; i < E; i += 32) hist[i] = 0;
        __syncwarp();
        int32_t cnt0 = 0, cnt1 = 0;  // this channel's tokens sent to rank lane / lane + 32
        for (int64_t t0 = b; t0 < e; t0 += 32) {
            const int64_t t = t0 + lane;
            const bool active = t < e;
            const int64_t g = s * a.T + t;
            int32_t ids[kMaxK];
#pragma unroll
            for (int k = 0; k < kMaxK; ++k) ids[k] = (k < K && active) ? __ldg(a.topk_idx + g * K + k) : -1;
            uint64_t mask = 0;
#pragma unroll
            for (int k = 0; k < kMaxK; ++k) {
                if (k < K) {
                    const int32_t ex = ids[k];
                    if (ex >= E) bad = true;
                    if (ex >= 0 && ex < E) {
                        atomicAdd(hist + ex, 1);  // integer counts: the order does not matter
                        mask |= 1ull << (ex / a.epr);
                    }
                }
            }
            if (active) {
                write_itr_row(a.itr + g * P, mask, P);
                if (a.bits)
                    for (int w = 0; w < W; ++w) a.bits[g * W + w] = static_cast<uint32_t>(mask >> (32 * w));
            }
            // Lanes over destinations: tokens of this step in order, so each
            // lane's running count is the token's position on its rank.
            const int m = e - t0 < 32 ? static_cast<int>(e - t0) : 32;
            int32_t* row = a.send_head + (s * a.T + t0) * P;
            for (int j = 0; j < m; ++j, row += P) {
                const unsigned long long mj = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(mask), j);
                const int32_t h0 = static_cast<int32_t>((mj >> lane) & 1ull);
                if (lane < P) row[lane] = h0 ? cnt0 : -1;
                cnt0 += h0;
                if (P > 32) {
                    const int32_t h1 = static_cast<int32_t>((mj >> (lane + 32)) & 1ull);
                    if (lane + 32 < P) row[lane + 32] = h1 ? cnt1 : -1;
                    cnt1 += h1;
                }
            }
        }
        if (lane < P) a.ccT[lane * a.PCp + ch] = cnt0;
        if (lane + 32 < P) a.ccT[(lane + 32) * a.PCp + ch] = cnt1;
        __syncwarp();
        for (int x = lane; x < E; x += 32) a.ecount[ch * E + x] = hist[x];
        __syncwarp();
    }
    return bad;
}

// ---- phase B: column scans (ranks) and expert sums ----------------------------------
// Skewed index into a warp's column copy: lane-contiguous runs of kSeg words
// fall in distinct banks.
__device__ __forceinline__ int64_t cx(int64_t j) { return j + (j >> 4); }

__device__ void scan_rank_column(const FusedArgs& a, int d, int32_t* colx, int lane) {
    const int P = a.P, C = a.C;
    const int64_t PC = a.PC;
    const int32_t* src = a.ccT + d * a.PCp;
    int32_t* rc = a.rcpm + d * PC;  // [d][s][c] with j = s * C + c
    int32_t carry = 0;
    for (int64_t j0 = 0; j0 < PC; j0 += 32 * kSeg) {
        const int64_t jb = j0 + static_cast<int64_t>(lane) * kSeg;
        int32_t v[kSeg];
#pragma unroll
        for (int q = 0; q < kSeg; q += 4) {
            // jb + q is a multiple of 4 and the row stride PCp too: whole int4 in the row.
            const int4 u = jb + q < a.PCp ? __ldcg(reinterpret_cast<const int4*>(src + jb + q)) : make_int4(0, 0, 0, 0);
            v[q] = u.x;
            v[q + 1] = u.y;
            v[q + 2] = u.z;
            v[q + 3] = u.w;
        }
        int32_t sum = 0;
#pragma unroll
        for (int u = 0; u < kSeg; ++u) {
            if (jb + u >= PC) v[u] = 0;  // row padding
            sum += v[u];
        }
        const int32_t incl = warp_incl_scan(sum, lane);
        int32_t run = carry + incl - sum;
#pragma unroll
        for (int u = 0; u < kSeg; ++u) {
            const int64_t j = jb + u;
            if (j < PC) {
                colx[cx(j)] = run;
                rc[j] = run;
            }
            run += v[u];
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) colx[cx(PC)] = carry;
    __syncwarp();
    for (int64_t j = lane; j < PC; j += 32) {
        const int64_t s = static_cast<uint32_t>(j) / static_cast<uint32_t>(C), c = j - s * C;
        a.cpm[(s * P + d) * C + c] = colx[cx(j + 1)] - colx[cx(s * C)];
    }
    for (int s = lane; s < P; s += 32) {
        const int32_t hi = colx[cx(static_cast<int64_t>(s + 1) * C)], lo = colx[cx(static_cast<int64_t>(s) * C)];
        a.ntpr[s * P + d] = hi - lo;
        a.rpm[s * P + d] = hi;
    }
    if (lane == 0) a.nrt[d] = carry;
    __syncwarp();
}

__device__ void sum_expert(const FusedArgs& a, int x, int lane) {
    const int C = a.C, E = a.E;
    int32_t tot = 0;
    for (int s = lane; s < a.P; s += 32) {
        const int32_t* src = a.ecount + static_cast<int64_t>(s) * C * E + x;
        int32_t sum = 0;
        for (int c0 = 0; c0 < C; c0 += kSumUnroll) {
            int32_t v[kSumUnroll];
#pragma unroll
            for (int u = 0; u < kSumUnroll; ++u)
                v[u] = c0 + u < C ? __ldcg(src + static_cast<int64_t>(c0 + u) * E) : 0;
#pragma unroll
            for (int u = 0; u < kSumUnroll; ++u) sum += v[u];
        }
        a.ntpe[static_cast<int64_t>(s) * E + x] = sum;
        tot += sum;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) a.nrtpe[x] = static_cast<int32_t>(round_up(tot, a.A));
}

__host__ __device__ __forceinline__ int64_t colx_words(int64_t PC) { return round_up(PC + (PC >> 4) + 2, 4); }

__device__ void phase_tables(const FusedArgs& a, int32_t* region) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* colx = region + warp * colx_words(a.PC);
    const int64_t total_warps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t tasks = static_cast<int64_t>(a.P) + a.E;
    for (int64_t task = static_cast<int64_t>(warp) * gridDim.x + blockIdx.x; task < tasks; task += total_warps) {
        if (task < a.P)
            scan_rank_column(a, static_cast<int>(task), colx, lane);
        else
            sum_expert(a, static_cast<int>(task - a.P), lane);
    }
}

// ---- phase C: payload -------------------------------------------------------------
// Channel of source-local token t (inverse of split_range over T = cq * C + cr
// tokens: channels below cr hold cq + 1 tokens, the others cq).
__device__ __forceinline__ uint32_t channel_of(uint32_t t, uint32_t cq, uint32_t cr) {
    const uint32_t big = cr * (cq + 1);
    return t < big ? t / (cq + 1) : cr + (t - big) / cq;
}

// Per-token routing a warp needs in phase C: for destinations lane and
// lane + 32 the local position (phase A, -1 if not sent) and the channel's
// first row on that rank (phase B); lane k < K holds slot k's expert and weight.
struct Route {
    int32_t loc[2], base[2], idx;
    float w;
    uint32_t s, t;  // source rank and source-local token
};

__device__ __forceinline__ void load_route(const FusedArgs& a, int64_t g, int lane, Route* r) {
    const uint32_t s = static_cast<uint32_t>(g) / static_cast<uint32_t>(a.T);
    const uint32_t t = static_cast<uint32_t>(g) - s * static_cast<uint32_t>(a.T);
    const int64_t ch = static_cast<int64_t>(s) * a.C + channel_of(t, a.cq, a.cr);
    r->s = s;
    r->t = t;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int dd = lane + 32 * h;
        r->loc[h] = dd < a.P ? __ldcg(a.send_head + g * a.P + dd) : -1;
        r->base[h] = dd < a.P ? __ldcg(a.rcpm + dd * a.PC + ch) : 0;
    }
    r->idx = lane < a.K ? __ldg(a.topk_idx + g * a.K + lane) : -1;
    r->w = (lane < a.K && a.topk_weights) ? __ldg(a.topk_weights + g * a.K + lane) : 0.f;
}

// Row buffers of one warp: token i of the warp's stream (g = first + i * step)
// goes to buffer i % NB, completing on bars[i % NB] with parity (i / NB) & 1.
struct Ring {
    uint64_t* bars;
    unsigned char* buf;
    int64_t first, step, n_local, last_issued;
};

__device__ __forceinline__ void ring_issue(const FusedArgs& a, Ring& r, int64_t i, uint32_t RB) {
    const int slot = static_cast<int>(i % a.nb);
    mbar_arrive_expect_tx(&r.bars[slot], RB);
    bulk_load(r.buf + static_cast<size_t>(slot) * RB, a.x + (r.first + i * r.step) * a.H, RB, &r.bars[slot]);
    r.last_issued = i;
}

// After an abort: wait (bounded) for this warp's loads still in flight, so no
// copy lands in shared memory after the CTA exits. Lane 0 only.
__device__ void ring_drain(const FusedArgs& a, Ring& r, int64_t first) {
    for (int64_t j = first; j <= r.last_issued; ++j)
        mbar_wait(&r.bars[j % a.nb], static_cast<uint32_t>((j / a.nb) & 1));
}

__device__ void phase_payload(const FusedArgs& a, Ring& ring, int64_t* prb) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = a.P, K = a.K, NB = a.nb;
    const DispatchArgs& d = a.d;
    const int64_t n_local = ring.n_local;
    const int64_t TW = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t gwarp = static_cast<int64_t>(warp) * gridDim.x + blockIdx.x;  // warp-major, as in phase A
    const uint32_t RB = static_cast<uint32_t>(a.H) * 2u;

    Route cur, nxt;
    if (n_local > 0) load_route(a, ring.first, lane, &cur);
    // part_row_base: exclusive scan of num_recv_tokens (64-bit), in every CTA.
    if (warp == 0) {
        int64_t run = 0;
        for (int d0 = 0; d0 < P; d0 += 32) {
            const int dd = d0 + lane;
            const int64_t v = dd < P ? __ldcg(a.nrt + dd) : 0;
            int64_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (dd < P) prb[dd] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) prb[P] = run;
        __syncwarp();
        if (blockIdx.x == 0)
            for (int dd = lane; dd <= P; dd += 32) a.part_row_base[dd] = prb[dd];
    }
    __syncthreads();
    // recv_expert_offset: one warp per rank, exclusive scan of its experts' aligned counts.
    for (int64_t dr = gwarp; dr < P; dr += TW) {
        int32_t carry = 0;
        for (int l0 = 0; l0 < a.epr; l0 += 32) {
            const int l = l0 + lane;
            const int32_t cnt = l < a.epr ? __ldcg(a.nrtpe + dr * a.epr + l) : 0;
            const int32_t incl = warp_incl_scan(cnt, lane);
            if (l < a.epr) a.reo[dr * a.epr + l] = carry + incl - cnt;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }

    bool failed = false;
    int64_t i = 0;
    for (; i < n_local; ++i) {
        const int slot = static_cast<int>(i % NB);
        const int64_t g = ring.first + i * ring.step;
        if (i + 1 < n_local) load_route(a, g + ring.step, lane, &nxt);
        // Global send_head rows for destinations lane and lane + 32.
        int32_t sh[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            sh[h] = cur.loc[h] >= 0 ? cur.loc[h] + cur.base[h] : -1;
            if (cur.loc[h] >= 0) a.send_head[g * P + lane + 32 * h] = sh[h];
        }
        const bool ok = mbar_wait(&ring.bars[slot], static_cast<uint32_t>((i / NB) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            failed = true;
            break;
        }
        const unsigned char* src = ring.buf + static_cast<size_t>(slot) * RB;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int dd = lane + 32 * h;
            if (sh[h] >= 0) {
                const int64_t lo = prb[dd], hi = prb[dd + 1], row = lo + sh[h];
                if (sh[h] < hi - lo && row >= 0 && row < d.arena_rows)
                    bulk_store(d.arena + row * d.stride, src, RB);
                else
                    raise_error(a.err, MOE_ERR_CAPACITY);
            }
        }
        bulk_commit();
        // Triple and side arrays of every destination row of token g.
        {
            const int32_t idx = cur.idx;
            const float w = cur.w;
            const int32_t dk = (idx >= 0 && idx < a.E) ? idx / a.epr : -1;
            const int32_t src_rank = static_cast<int32_t>(cur.s), src_tok = static_cast<int32_t>(cur.t);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t todo = __ballot_sync(0xffffffffu, sh[h] >= 0);
                while (todo) {
                    const int j = __ffs(todo) - 1;
                    todo &= todo - 1;
                    const int dj = j + 32 * h;
                    const int32_t shd = __shfl_sync(0xffffffffu, sh[h], j);
                    const int64_t lo = prb[dj], hi = prb[dj + 1], row = lo + shd;
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
        // Refill: with two or more buffers, token i-1's buffer (its stores have
        // left shared memory once at most one group, token i's, still reads);
        // with one buffer, token i's own.
        int64_t done_tok;
        if (NB >= 2) {
            bulk_wait_read<1>();
            done_tok = i - 1;
        } else {
            bulk_wait_read<0>();
            done_tok = i;
        }
        __syncwarp();
        if (lane == 0 && done_tok >= 0 && done_tok + NB < n_local) ring_issue(a, ring, done_tok + NB, RB);
        __syncwarp();
        cur = nxt;
    }
    bulk_wait<0>();
    if (failed && lane == 0) {
        raise_error(a.err, MOE_ERR_DEVICE_TIMEOUT);
        ring_drain(a, ring, i);
    }
}

// Zeroes the grid barrier counter. Launched just before fused_kernel with
// programmatic stream serialisation: it lets fused_kernel be scheduled at once,
// then waits for the previous work on the stream before the store; fused_kernel
// waits for this grid to complete before it touches global memory.
__global__ void fused_prep_kernel(unsigned int* counter) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) *counter = 0u;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) fused_kernel(const FusedArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_wait_then_release();
    MOE_PROF_BEGIN(kProfFused);
    __shared__ int64_t prb[kMaxP + 1];
    const unsigned int n = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t RB = static_cast<uint32_t>(a.H) * 2u;
    int32_t* region = reinterpret_cast<int32_t*>(smem + a.ab_off);

    // Start the row loads of each warp's first tokens: they overlap phases A and B.
    Ring ring;
    ring.bars = reinterpret_cast<uint64_t*>(smem) + warp * kMaxNB;
    ring.buf = smem + kBarBytes + static_cast<size_t>(warp) * a.nb * RB;
    // Tokens are dealt to CTAs first (g mod gridDim), so every SM -- whose
    // bulk-copy engine all its warps share -- gets the same number of rows.
    ring.first = blockIdx.x + static_cast<int64_t>(n) * warp;
    ring.step = static_cast<int64_t>(n) * kWarps;
    ring.n_local = ring.first < a.S ? (a.S - 1 - ring.first) / ring.step + 1 : 0;
    ring.last_issued = -1;
    if (lane == 0) {
        for (int b = 0; b < a.nb; ++b) mbar_init(&ring.bars[b], 1);
        mbar_init_fence();
        const int64_t npro = ring.n_local < a.nb ? ring.n_local : a.nb;
        for (int64_t i = 0; i < npro; ++i) ring_issue(a, ring, i, RB);
    }
    __syncwarp();

    // err starts at 0: CTA 0 clears it before the first grid barrier, and every
    // status is raised after that barrier.
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.err) *a.err = 0;
    const bool bad = __syncthreads_or(phase_counts(a, region));
    MOE_STAMP(1);
    bool ok = grid_barrier(a.barrier, n, a.err, a.spin_limit, blockIdx.x == a.skip_arrival);
    MOE_STAMP(2);
    if (ok) {
        if (bad && threadIdx.x == 0) raise_error(a.err, MOE_ERR_TOPK_OUT_OF_RANGE);
        phase_tables(a, region);
        MOE_STAMP(3);
        ok = grid_barrier(a.barrier, 2 * n, a.err, a.spin_limit, false);
        MOE_STAMP(4);
    }
    if (!ok) {
        if (lane == 0) ring_drain(a, ring, 0);
        MOE_PROF_END();
        return;
    }
    phase_payload(a, ring, prb);
    MOE_STAMP(5);
    MOE_PROF_END();
}

// The next moe_dispatch_fused call of this host thread, when armed by
// moe_test_fused_barrier: grid-barrier spin limit and the CTA that leaves out
// its first arrival.
thread_local uint32_t t_test_spin_limit = 0;
thread_local int64_t t_test_skip_cta = -1;

// Row buffers per warp, the offset of the phase A / B region and the dynamic
// shared memory of the launch, for a budget of `limit` bytes.
// Per device: 0 = not tried yet, 1 = cooperative + programmatic serialisation
// accepted, 2 = refused.
std::atomic<int> g_coop_pdl[64];

void fused_plan(const moe_shape& s, int64_t limit, int* nb, uint32_t* ab_off, size_t* smem) {
    const int64_t pc = static_cast<int64_t>(s.P) * s.num_channels;
    const int64_t a = static_cast<int64_t>(kWarps) * s.E * 4;
    const int64_t b = static_cast<int64_t>(kWarps) * colx_words(pc) * 4;
    const int64_t ab = a > b ? a : b;
    const int64_t rb = static_cast<int64_t>(s.H) * 2;
    const int64_t avail = limit - kBarBytes - ab;
    int64_t n = avail > 0 ? avail / (kWarps * rb) : 0;
    n = n > kMaxNB ? kMaxNB : n;
    *nb = static_cast<int>(n);
    *ab_off = static_cast<uint32_t>(kBarBytes + kWarps * n * rb);
    *smem = static_cast<size_t>(*ab_off + ab);
}

}  // namespace

void arm_fused_barrier_test(uint32_t spin_limit, int64_t skip_cta) {
    t_test_spin_limit = spin_limit;
    t_test_skip_cta = skip_cta;
}

bool fused_supported(const moe_shape& s) {
    if (!(s.P <= kMaxP && s.E <= kMaxE && s.H <= kMaxH && s.K <= kMaxK && s.quant == 0 &&
          static_cast<int64_t>(s.P) * s.num_channels <= kMaxPC))
        return false;
    int nb = 0;
    uint32_t off = 0;
    size_t smem = 0;
    fused_plan(s, kSmemBudget, &nb, &off, &smem);
    return nb >= 1;
}

int64_t fused_scratch_bytes(const moe_shape& s) {
    const int64_t pc = static_cast<int64_t>(s.P) * s.num_channels;
    return round_up(256 + (static_cast<int64_t>(s.P) * round_up(pc, 4) + pc * s.E) * 4, 256);
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
    a.PC = static_cast<int64_t>(s.P) * s.num_channels;
    a.PCp = round_up(a.PC, 4);
    a.cq = static_cast<uint32_t>(a.T / s.num_channels);
    a.cr = static_cast<uint32_t>(a.T % s.num_channels);
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
    unsigned char* sc = static_cast<unsigned char*>(scratch);
    a.barrier = reinterpret_cast<unsigned int*>(sc);
    a.ccT = reinterpret_cast<int32_t*>(sc + 256);
    a.ecount = a.ccT + a.PCp * s.P;
    a.err = err;
    a.spin_limit = kSpinLimit;
    a.skip_arrival = -1;
    if (t_test_spin_limit != 0) {  // one call armed by moe_test_fused_barrier
        a.spin_limit = t_test_spin_limit;
        a.skip_arrival = t_test_skip_cta;
        t_test_spin_limit = 0;
        t_test_skip_cta = -1;
    }
    const int static_smem = kernel_static_smem(reinterpret_cast<const void*>(fused_kernel));
    if (static_smem < 0) return cudaErrorInvalidDeviceFunction;
    int64_t limit = static_cast<int64_t>(device_optin_smem()) - static_smem;
    if (limit > kSmemBudget) limit = kSmemBudget;
    size_t smem = 0;
    // The most CTAs per SM (up to kCtasPerSm) whose share of the SM's shared
    // memory, less the per-CTA reservation, holds a row buffer per warp.
    int cps = kCtasPerSm;
    for (; cps > 1; --cps) {
        int64_t share = static_cast<int64_t>(device_sm_smem()) / cps - 1024 - static_smem;
        if (share > limit) share = limit;
        fused_plan(s, share, &a.nb, &a.ab_off, &smem);
        if (a.nb >= 1) break;
    }
    if (cps == 1) fused_plan(s, limit, &a.nb, &a.ab_off, &smem);
    if (a.nb < 1) return cudaErrorInvalidConfiguration;
    int per_sm = 0;
    cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(fused_kernel), smem, kThreads, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (per_sm < cps) cps = per_sm;
    // cps CTAs per SM, all resident at once (cooperative launch).
    const int grid = device_sm_count() * cps;
    e = launch_pdl(fused_prep_kernel, 1, 32, 0, stream, a.barrier);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // Whether this device takes a cooperative launch with programmatic
    // serialisation is learnt on the first call and remembered, so a refusal is
    // not paid again on every call. Without it the launch simply follows the
    // prep kernel.
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool slot = dev >= 0 && dev < 64;
    const int known = slot ? g_coop_pdl[dev].load(std::memory_order_relaxed) : 0;
    if (known != 2) {
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, fused_kernel, a);
        if (e == cudaSuccess) {
            if (slot) g_coop_pdl[dev].store(1, std::memory_order_relaxed);
            return e;
        }
        // Only a refusal of the attribute combination itself is remembered;
        // any other failure (e.g. too large for the SMs free right now, or an
        // error left by earlier work) is returned, and the next call tries again.
        if (known == 1 || (e != cudaErrorNotSupported && e != cudaErrorInvalidValue)) return e;
        (void)cudaGetLastError();  // clears this launch's own refusal
        if (slot) g_coop_pdl[dev].store(2, std::memory_order_relaxed);
    }
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_kernel, a);
}

MOE_PROFILE_UNIT(fused)

}  // namespace moe
