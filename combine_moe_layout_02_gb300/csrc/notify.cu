// notify.cu -- counts and prefixes (moe_notify).
//
// "Ascend DeepEP MoE Dispatch Optimization", section "Notify 先交换数量和前缀":
// notify turns the routing into how many rows each rank receives, how many per
// local expert, and where each (source rank, channel) segment starts. Section
// "Device 侧如何把 channel 变成远端 Put" gives the receive position of a row:
// rank_prefix_matrix[s-1][d] + channel_prefix_matrix[s][d][c-1] + the running
// count inside channel c. "internode.cu", section 1 (notify_dispatch) rounds
// the per-expert receive counts up to expert_alignment. Channel c of a source
// rank is the c-th block of the balanced split of "HCCL Window 模式
// (Non-SHMEM) 代码深度剖析", section 8.3.
//
// The receive position of token g of source rank s on rank d unrolls to
//   rank_prefix[s-1][d] + (tokens of s before g that are bound for d):
// the channels only cut that running count into the matrices' segments. So
// every output of a source rank follows from its own rows of
// is_token_in_rank plus sums of num_tokens_per_rank / num_tokens_per_expert,
// and one launch suffices: one thread-block cluster per source rank s, with
// no synchronisation between clusters.
//
// Inside the cluster each warp takes a contiguous segment of s's tokens.
// Lanes are laid out as (token, group of 4 ranks): for P/4 <= 32 groups a
// token takes L = the next power of two >= P/4 lanes and a warp covers 32/L
// tokens per step (16 at P = 8, 1 at P = 128); each lane loads the token's 4
// flags of its group as one 32-bit word.
//  1. Count: each warp counts its segment's tokens per rank.
//  2. Block: per-warp counts become exclusive warp offsets and CTA totals;
//     cluster barrier; each CTA adds the totals of the CTAs before it
//     (distributed shared memory) -- the segment bases.
//  3. Heads: each warp walks its segment again; the 4 flags of a lane are
//     packed one per byte, so one shuffle scan over the token lanes gives
//     the exclusive counts of 4 ranks at once. send_head rows are written
//     as 16-byte stores; a token that starts a channel writes that
//     channel's recv_channel_prefix_matrix entry and the previous channel's
//     channel_prefix_matrix entry.
// Beside the scan, the cluster adds up rank_prefix_matrix's column prefix
// over the earlier source ranks (split over its CTAs), and cluster s sums the
// per-expert counts of rank s (num_recv_tokens_per_expert, recv_expert_offset);
// cluster P-1 also writes num_recv_tokens and the packed partition bases.
// No atomics: every output is a fixed-order integer sum.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kNotifyThreads = 256;
constexpr int kNotifyWarps = kNotifyThreads / 32;
constexpr int kNotifyMaxCluster = 16;

constexpr int kNotifyCache = 4;          // flag words a lane keeps in registers between the passes
static_assert(kNotifyCache == 4, "the second pass selects among exactly four cached words");
constexpr int kNotifyChanBuf = 4096;     // int32 entries of the channel-start buffer
constexpr int kNotifySmemSteps = 16;     // steps per warp whose flags shared memory can keep

struct NotifySmem {
    size_t wcnt, xc, xr, tmp_r, base, total, rprev, ecnt, chv, fsm, bytes;
};

// Shared memory (int32 unless noted): wcnt [warps][P]; xc, xr [cs][P] (the
// cluster CTAs' totals and rank-prefix partials; this CTA's own row is the
// one peers read); tmp_r [threads] int4; base [P];
// total [P]; rprev [P]; ecnt [E/P]; chv [channels starting
// in this CTA's tokens][P] when that fits kNotifyChanBuf; with fsteps > 0,
// fsm uint32 [warps][fsteps][32]: each lane's flag words between the passes.
__host__ __device__ inline NotifySmem notify_smem(int P, int E, int cs, int fsteps) {
    NotifySmem m;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += (bytes + 15) / 16 * 16;
        return at;
    };
    m.wcnt = take(static_cast<size_t>(kNotifyWarps) * P * 4);
    m.xc = take(static_cast<size_t>(cs) * P * 4);
    m.xr = take(static_cast<size_t>(cs) * P * 4);
    m.tmp_r = take(kNotifyThreads * 16);
    m.base = take(static_cast<size_t>(P) * 4);
    m.total = take(static_cast<size_t>(P) * 4);
    m.rprev = take(static_cast<size_t>(P) * 4);
    m.ecnt = take(static_cast<size_t>(E / P) * 4);
    m.chv = take(kNotifyChanBuf * 4);
    m.fsm = take(static_cast<size_t>(kNotifyWarps) * fsteps * 32 * 4);
    m.bytes = o;
    return m;
}

template <typename V>
__device__ __forceinline__ V warp_inclusive_scan(V v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Each byte of w that is nonzero becomes 1, the others 0.
__device__ __forceinline__ uint32_t nz_bytes(uint32_t w) {
    uint32_t t = w | (w >> 4);
    t |= t >> 2;
    t |= t >> 1;
    return t & 0x01010101u;
}

__device__ __forceinline__ int byte_of(uint32_t w, int j) { return static_cast<int>((w >> (8 * j)) & 0xffu); }

// Flags of ranks d..d+3 of row `row` (one per byte, 0/1); ranks >= P give 0.
template <bool A4>
__device__ __forceinline__ uint32_t load_flags(const uint8_t* row, int d, int P) {
    if (A4) return nz_bytes(__ldg(reinterpret_cast<const uint32_t*>(row + d)));
    uint32_t f = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (d + j < P && __ldg(row + d + j) != 0) f |= 1u << (8 * j);
    return f;
}

// First token of channel c under the balanced split of T tokens over C
// channels (q = T / C, rr = T % C; begin(C) = T).
__device__ __forceinline__ int32_t channel_begin(int32_t c, int32_t q, int32_t rr) {
    return c * q + min(c, rr);
}

// floor(n / d) for 0 <= n < 2^31 and 1 <= d < 2^31, with m = div_magic(d) =
// ceil(2^32 / d) from the host: the multiply-shift estimate is the quotient
// or one more (the error term is below n / 2^32 < 1/2), so one correction.
__device__ __forceinline__ int32_t div_m(int32_t n, int32_t d, uint64_t m) {
    uint32_t q = static_cast<uint32_t>((static_cast<uint64_t>(static_cast<uint32_t>(n)) * m) >> 32);
    if (q * static_cast<uint32_t>(d) > static_cast<uint32_t>(n)) --q;
    return static_cast<int32_t>(q);
}
inline uint64_t div_magic(int32_t d) {
    const uint64_t dd = static_cast<uint64_t>(d < 1 ? 1 : d);
    return ((uint64_t{1} << 32) + dd - 1) / dd;
}

// The first channel that starts at or after token t < T; m1 = div_magic(q + 1),
// m0 = div_magic(q) (q >= 1 whenever t >= rr * (q + 1)).
__device__ __forceinline__ int32_t next_channel(int32_t t, int32_t q, int32_t rr, uint64_t m1, uint64_t m0) {
    const int32_t bnd = rr * (q + 1);  // tokens in the rr longer channels
    int32_t c = t < bnd ? div_m(t, q + 1, m1) : rr + div_m(t - bnd, q, m0);
    if (channel_begin(c, q, rr) < t) ++c;
    return c;
}

// Shape constants of a launch, split on the host so that the kernel does no
// integer division: T = tokens per source rank; cs = CTAs per cluster (a
// power of two, 2^lcs); the warps' token segments are the balanced split of
// T over cs * kNotifyWarps (wq, wr); the channels that of T over C (cq, cr);
// each CTA sums a balanced share of rank s's E/P experts (eq, er).
struct NotifyParams {
    int32_t P, E, C, A, epr, T, cs, lcs;
    int32_t wq, wr, cq, cr, eq, er;
    const int32_t* ntpr;
    const int32_t* ntpe;
    const uint8_t* itr;
    int32_t *rpm, *cpm, *rcpm, *nrt, *nrtpe, *reo, *send_head;
    int64_t* part_row_base;
    int32_t fsteps;     // kNotifySmemSteps when the flags are kept in shared memory, else 0
    uint64_t mq1, mq0;  // div_magic(cq + 1), div_magic(cq)
    // notify_small_kernel only: log2 of the lanes per token, rows of the two
    // partial-sum tables, division constants, shared-memory offsets (bytes)
    int32_t lg, sR, sRq;
    uint64_t mP, mE, mA;
    int32_t off_wcnt, off_rpart, off_epart, off_rprev, off_total, off_ecnt, off_chv;
};

// Grid: P clusters of cs CTAs of kNotifyThreads threads; cluster s handles
// source rank s.
template <bool A4>
__global__ void __launch_bounds__(kNotifyThreads, 4) notify_kernel(const NotifyParams a) {
    pdl_wait_then_release();
    MOE_PROF_BEGIN(kProfNotify);
    extern __shared__ __align__(16) unsigned char smem[];
    const int32_t P = a.P, E = a.E, C = a.C, A = a.A;
    const int32_t T = a.T;
    const int32_t* __restrict__ ntpr = a.ntpr;
    const int32_t* __restrict__ ntpe = a.ntpe;
    const uint8_t* __restrict__ itr = a.itr;
    int32_t* __restrict__ rpm = a.rpm;
    int32_t* __restrict__ cpm = a.cpm;
    int32_t* __restrict__ rcpm = a.rcpm;
    int32_t* __restrict__ nrt = a.nrt;
    int32_t* __restrict__ nrtpe = a.nrtpe;
    int32_t* __restrict__ reo = a.reo;
    int32_t* __restrict__ send_head = a.send_head;
    int64_t* __restrict__ part_row_base = a.part_row_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cs = a.cs;
    const int r = static_cast<int>(cluster_ctarank());
    const int32_t s = static_cast<int32_t>(cluster_id_x());
    const NotifySmem M = notify_smem(P, E, cs, a.fsteps);
    int32_t* wcnt = reinterpret_cast<int32_t*>(smem + M.wcnt);
    int32_t* xc = reinterpret_cast<int32_t*>(smem + M.xc);
    int32_t* xr = reinterpret_cast<int32_t*>(smem + M.xr);
    int4* tmp_r = reinterpret_cast<int4*>(smem + M.tmp_r);
    int32_t* base = reinterpret_cast<int32_t*>(smem + M.base);
    int32_t* total = reinterpret_cast<int32_t*>(smem + M.total);
    int32_t* rprev = reinterpret_cast<int32_t*>(smem + M.rprev);
    int32_t* ecnt = reinterpret_cast<int32_t*>(smem + M.ecnt);
    int32_t* chv = reinterpret_cast<int32_t*>(smem + M.chv);
    uint32_t* fsm = reinterpret_cast<uint32_t*>(smem + M.fsm);
    int32_t* ctot = xc + r * P;   // this CTA's totals (read by the peers)
    int32_t* rpart = xr + r * P;  // this CTA's rank-prefix partial (read by the peers)

    const int epr = a.epr;
    const int G = (P + 3) >> 2;  // rank groups of 4
    const int32_t gw = r * kNotifyWarps + warp;
    const int32_t sb = gw * a.wq + min(gw, a.wr);
    const int32_t se = sb + a.wq + (gw < a.wr ? 1 : 0);
    const int32_t cq = a.cq, cr = a.cr;
    const uint8_t* src_rows = itr + static_cast<int64_t>(s) * T * P;

    // --- every load that does not wait on another, issued first -----------
    // (a) rank-prefix partial: rows [pb, pe) of the source ranks before s,
    //     4 ranks per thread (A4) and rpp rows per pass.
    const int32_t sq = s >> a.lcs, sr = s & (cs - 1);
    const int32_t pb = r * sq + min(r, sr);
    const int32_t pe = pb + sq + (r < sr ? 1 : 0);
    const int cols = A4 ? P >> 2 : P;
    const int rpp = max(1, min(cols >= kNotifyThreads ? 1 : kNotifyThreads / cols, pe - pb));
    int4 racc = make_int4(0, 0, 0, 0);
    if (cols <= kNotifyThreads && tid < rpp * cols) {
        const int cg = tid % cols;
#pragma unroll 8
        for (int32_t q = pb + tid / cols; q < pe; q += rpp) {
            if (A4) {
                const int4 v = __ldg(reinterpret_cast<const int4*>(ntpr + static_cast<int64_t>(q) * P) + cg);
                racc.x += v.x;
                racc.y += v.y;
                racc.z += v.z;
                racc.w += v.w;
            } else {
                racc.x += __ldg(ntpr + static_cast<int64_t>(q) * P + cg);
            }
        }
    }
    // (b) receive counts of rank s's experts: this CTA's share [lb, le) of
    //     them, one warp per expert (the first 8 loaded here), lanes over the
    //     source ranks.
    const int32_t lb = r * a.eq + min(r, a.er);
    const int32_t le = lb + a.eq + (r < a.er ? 1 : 0);
    const int32_t* ecol = ntpe + static_cast<int64_t>(s) * epr;  // rank s's experts in row 0
    int32_t esum = 0;
    if (lb + warp < le)
        for (int q = lane; q < P; q += 32) esum += __ldg(ecol + static_cast<int64_t>(q) * E + lb + warp);
    // --- 1. count ---------------------------------------------------------
    // With one block of rank groups and at most kNotifyCache steps per warp,
    // a lane's flag words stay in registers for the second pass; with up to
    // kNotifySmemSteps steps (a.fsteps > 0), in shared memory, all loaded at
    // once.
    uint32_t fc[kNotifyCache];
    bool cached = false;
    const bool scached = a.fsteps > 0;
    uint32_t* fs = fsm + warp * (kNotifySmemSteps * 32) + lane;
    for (int rb = 0; rb * 32 < G; ++rb) {
        const int gn = min(32, G - rb * 32);
        int L = 1;
        while (L < gn) L <<= 1;
        const int tpw = 32 / L;
        const int g = lane & (L - 1), tk = lane / L;
        const int d = 4 * (rb * 32 + g);
        int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
        cached = G <= 32 && se - sb <= kNotifyCache * tpw;
        if (cached) {
#pragma unroll
            for (int i = 0; i < kNotifyCache; ++i) {
                const int32_t t = sb + tk + i * tpw;
                fc[i] = (g < gn && t < se) ? load_flags<A4>(src_rows + static_cast<int64_t>(t) * P, d, P) : 0u;
            }
#pragma unroll
            for (int i = 0; i < kNotifyCache; ++i) {
                c0 += byte_of(fc[i], 0);
                c1 += byte_of(fc[i], 1);
                c2 += byte_of(fc[i], 2);
                c3 += byte_of(fc[i], 3);
            }
        } else if (scached) {
#pragma unroll 8
            for (int i = 0; i < kNotifySmemSteps; ++i) {
                const int32_t t = sb + tk + i * tpw;
                const uint32_t f =
                    (g < gn && t < se) ? load_flags<A4>(src_rows + static_cast<int64_t>(t) * P, d, P) : 0u;
                fs[i * 32] = f;
                c0 += byte_of(f, 0);
                c1 += byte_of(f, 1);
                c2 += byte_of(f, 2);
                c3 += byte_of(f, 3);
            }
        } else if (g < gn) {
#pragma unroll 4
            for (int32_t t = sb + tk; t < se; t += tpw) {
                const uint32_t f = load_flags<A4>(src_rows + static_cast<int64_t>(t) * P, d, P);
                c0 += byte_of(f, 0);
                c1 += byte_of(f, 1);
                c2 += byte_of(f, 2);
                c3 += byte_of(f, 3);
            }
        }
        for (int o = L; o < 32; o <<= 1) {
            c0 += __shfl_xor_sync(0xffffffffu, c0, o);
            c1 += __shfl_xor_sync(0xffffffffu, c1, o);
            c2 += __shfl_xor_sync(0xffffffffu, c2, o);
            c3 += __shfl_xor_sync(0xffffffffu, c3, o);
        }
        if (tk == 0 && g < gn) {
            int32_t* wc = wcnt + warp * P + d;
            wc[0] = c0;
            if (d + 1 < P) wc[1] = c1;
            if (d + 2 < P) wc[2] = c2;
            if (d + 3 < P) wc[3] = c3;
        }
    }
    if (cols <= kNotifyThreads && tid < rpp * cols) tmp_r[tid] = racc;
    MOE_STAMP(1);
    __syncthreads();
    MOE_STAMP(2);

    // --- 2. block totals, exclusive warp offsets, partials -----------------
    for (int d = tid; d < P; d += kNotifyThreads) {
        int32_t run = 0;
        for (int w = 0; w < kNotifyWarps; ++w) {
            const int32_t v = wcnt[w * P + d];
            wcnt[w * P + d] = run;
            run += v;
        }
        ctot[d] = run;
        int32_t rp = 0;
        if (cols <= kNotifyThreads) {
            const int cg = A4 ? d >> 2 : d, j = A4 ? d & 3 : 0;
            for (int k = 0; k < rpp; ++k) {
                const int4 v = tmp_r[k * cols + cg];
                rp += j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
            }
        } else {
            for (int32_t q = pb; q < pe; ++q) rp += __ldg(ntpr + static_cast<int64_t>(q) * P + d);
        }
        rpart[d] = rp;
    }
    for (int32_t l = lb + warp; l < le; l += kNotifyWarps) {
        int32_t sum = esum;
        if (l != lb + warp) {
            sum = 0;
            for (int q = lane; q < P; q += 32) sum += __ldg(ecol + static_cast<int64_t>(q) * E + l);
        }
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) ecnt[l] = (sum + A - 1) / A * A;  // fits int32 (shape limits)
    }
    MOE_STAMP(3);
    cluster_sync_all();
    MOE_STAMP(4);
    // Every (rank, peer CTA) pair read by its own thread, then summed locally.
    for (int i = tid; i < P * cs; i += kNotifyThreads) {
        const int q = i / P, d = i - q * P;
        if (q != r) {
            xc[q * P + d] = ld_cluster_s32(cluster_map(xc + q * P + d, q));
            xr[q * P + d] = ld_cluster_s32(cluster_map(xr + q * P + d, q));
        }
    }
    if (r == 0 && warp == kNotifyWarps - 1) {
        // Rank s's per-expert counts from the CTAs that summed them, scanned.
        const int32_t eq = a.eq, er = a.er;
        int32_t carry = 0;
        for (int l0 = 0; l0 < epr; l0 += 32) {
            const int l = l0 + lane;
            int32_t v = 0;
            if (l < epr) {
                const int owner = l < er * (eq + 1) ? l / (eq + 1) : er + (l - er * (eq + 1)) / eq;
                v = owner == 0 ? ecnt[l] : ld_cluster_s32(cluster_map(ecnt + l, owner));
            }
            const int32_t incl = warp_inclusive_scan(v, lane);
            if (l < epr) {
                nrtpe[s * epr + l] = v;
                reo[s * epr + l] = carry + incl - v;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    cluster_arrive();  // done reading the peers; their shared memory may go at the final wait
    __syncthreads();
    for (int d = tid; d < P; d += kNotifyThreads) {
        int32_t before = 0, all = 0, rp = 0;
#pragma unroll 4
        for (int q = 0; q < cs; ++q) {
            const int32_t v = xc[q * P + d];
            before += q < r ? v : 0;
            all += v;
            rp += xr[q * P + d];
        }
        base[d] = before;
        total[d] = all;
        rprev[d] = rp;
    }
    __syncthreads();
    MOE_STAMP(5);

    // --- per-rank outputs (from the prefixes and totals alone) -----------
    if (r == cs - 1) {
        // Channels that end at T (the last, and empty trailing ones when T < C)
        // and channels that start at T (empty ones).
        const int32_t cl = T < C ? (T > 0 ? T - 1 : 0) : C - 1;
        const int32_t cb = T < C ? T : C;
        for (int d = tid; d < P; d += kNotifyThreads) {
            const int32_t tot = total[d], rp = rprev[d];
            rpm[s * P + d] = rp + tot;
            for (int32_t c = cl; c < C; ++c) cpm[(static_cast<int64_t>(s) * P + d) * C + c] = tot;
            for (int32_t c = cb; c < C; ++c) rcpm[(static_cast<int64_t>(d) * P + s) * C + c] = rp + tot;
            if (s == P - 1) nrt[d] = rp + tot;
        }
    }
    if (s == P - 1 && r == 0 && warp == 0) {
        // Packed partition bases: the exclusive scan of the receive totals.
        int64_t run = 0;
        for (int d0 = 0; d0 < P; d0 += 32) {
            const int dd = d0 + lane;
            const int64_t v = dd < P ? static_cast<int64_t>(rprev[dd]) + total[dd] : 0;
            const int64_t incl = warp_inclusive_scan(v, lane);
            if (dd < P) part_row_base[dd] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) part_row_base[P] = run;
    }

    // --- 3. heads ------------------------------------------------------------
    // Channels that start inside this CTA's tokens [cta_b, cta_e): their
    // counts go to chv (written out coalesced below) when they fit.
    const int32_t cta_b = r * kNotifyWarps * a.wq + min(r * kNotifyWarps, a.wr);
    const int32_t cta_e = min(T, cta_b + kNotifyWarps * a.wq + max(0, min(kNotifyWarps, a.wr - r * kNotifyWarps)));
    const int32_t nonempty = min(T, C);  // channels that start before T
    const int32_t c_lo = cta_b < T ? next_channel(cta_b, cq, cr, a.mq1, a.mq0) : nonempty;
    const int32_t c_hi = cta_e < T ? next_channel(cta_e, cq, cr, a.mq1, a.mq0) : nonempty;
    const bool buffered = static_cast<int64_t>(c_hi - c_lo) * P <= kNotifyChanBuf;
    for (int rb = 0; rb * 32 < G; ++rb) {
        const int gn = min(32, G - rb * 32);
        int L = 1;
        while (L < gn) L <<= 1;
        const int tpw = 32 / L;
        const int g = lane & (L - 1), tk = lane / L;
        const int d = 4 * (rb * 32 + g);
        const bool gvalid = g < gn;
        const int last = (tpw - 1) * L + g;  // lane of this group's last token in a step
        int run[4], rp[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool ok = gvalid && d + j < P;
            run[j] = ok ? base[d + j] + wcnt[warp * P + d + j] : 0;
            rp[j] = ok ? rprev[d + j] : 0;
        }
        // Next channel start at or after this lane's token (nb = T: none).
        int32_t nc = sb + tk < se ? next_channel(sb + tk, cq, cr, a.mq1, a.mq0) : C;
        int32_t nb = channel_begin(nc, cq, cr);
        MOE_STAMP(8);
        // One step: tpw tokens, this lane's token t and flags f.
        auto step = [&](int32_t t, uint32_t f) {
            const bool tv = gvalid && t < se;
            // Inclusive counts over this step's tokens, 4 ranks per word.
            uint32_t incl = f;
            for (int o = L; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const uint32_t excl = incl - f;
            const uint32_t step_total = L == 32 ? f : __shfl_sync(0xffffffffu, incl, last);
            if (tv) {
                int loc[4], v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    loc[j] = run[j] + byte_of(excl, j);
                    v[j] = byte_of(f, j) ? rp[j] + loc[j] : -1;
                }
                int32_t* out = send_head + (static_cast<int64_t>(s) * T + t) * P + d;
                if (A4) {
                    *reinterpret_cast<int4*>(out) = make_int4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (d + j < P) out[j] = v[j];
                }
                while (nb < t) nb = channel_begin(++nc, cq, cr);
                if (nb == t) {  // t starts channel nc
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (d + j < P) {
                            if (buffered) {
                                chv[(nc - c_lo) * P + d + j] = loc[j];
                            } else {
                                rcpm[(static_cast<int64_t>(d + j) * P + s) * C + nc] = rp[j] + loc[j];
                                if (nc > 0) cpm[(static_cast<int64_t>(s) * P + d + j) * C + nc - 1] = loc[j];
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) run[j] += byte_of(step_total, j);
        };
        // One copy of the step code. The flags come from the registers of the
        // count pass (selected without indexing) or, when the segment is
        // longer, are read again kNotifyCache steps at a time, so that the
        // loads of four steps are in flight together rather than one L2 round
        // trip per step.
#pragma unroll 1
        for (int32_t i = 0, t0 = sb; t0 < se; ++i, t0 += tpw) {
            const int k = i & (kNotifyCache - 1);
            if (scached) {
                step(t0 + tk, fs[i * 32]);
                continue;
            }
            if (!cached && k == 0) {
#pragma unroll
                for (int j = 0; j < kNotifyCache; ++j) {
                    const int32_t tj = t0 + j * tpw + tk;
                    fc[j] = (gvalid && tj < se) ? load_flags<A4>(src_rows + static_cast<int64_t>(tj) * P, d, P) : 0u;
                }
            }
            const uint32_t f = k == 0 ? fc[0] : (k == 1 ? fc[1] : (k == 2 ? fc[2] : fc[3]));
            step(t0 + tk, f);
        }
    }
    MOE_STAMP(9);
    if (buffered) {
        __syncthreads();
        MOE_STAMP(10);
        // recv_channel_prefix_matrix[d][s][c] and channel_prefix_matrix[s][d][c-1]
        // for the channels starting here: c runs fastest, so consecutive
        // threads write consecutive entries of a row.
        const int nch = c_hi - c_lo;
        for (int i = tid; i < nch * P; i += kNotifyThreads) {
            const int d = i / nch, k = i - d * nch;
            const int32_t c = c_lo + k;
            const int32_t v = chv[k * P + d];
            rcpm[(static_cast<int64_t>(d) * P + s) * C + c] = rprev[d] + v;
            if (c > 0) cpm[(static_cast<int64_t>(s) * P + d) * C + c - 1] = v;
        }
    }

    MOE_STAMP(6);
    cluster_wait();
    MOE_STAMP(7);
    MOE_PROF_END();
}

// ---------------------------------------------------------------------------
// Small source ranks: one CTA of kSmallThreads threads holds all T tokens of
// rank s (each warp's tokens in at most kNotifyCache steps), so no cluster
// exchange is needed. Every reduction is a warp of lanes with shuffles, run
// side by side after one block barrier:
//   - per rank d, the exclusive offsets of the warps' counts (lane = warp);
//   - per rank d, the column sum of num_tokens_per_rank over the source ranks
//     before s (partial sums of kSmallThreads / P rows each, then the lanes);
//   - per local expert l, the sum of num_tokens_per_expert[.][s * E/P + l] over
//     the source ranks, rounded up to expert_alignment.
// The heads pass and the channel matrices follow the cluster kernel above.
// 512 threads measured fastest on GB300 (p32_e256_t128: front 10.8 us at
// 512, 12.0 at 1024, 12.9 at 256; tiny_p4_e16: 7.8, 8.9, 7.5): more warps
// repeat the per-warp set-up, fewer lengthen each warp's chain.
#ifndef MOE_NOTIFY_SMALL_THREADS
#define MOE_NOTIFY_SMALL_THREADS 512
#endif
constexpr int kSmallThreads = MOE_NOTIFY_SMALL_THREADS;
constexpr int kSmallWarps = kSmallThreads / 32;
static_assert(kSmallWarps <= 32 && kSmallThreads % 32 == 0, "the warp-offset scan puts one warp per lane");

struct SmallSmem {
    size_t wcnt, rpart, epart, rprev, total, ecnt, chv, bytes;
};

// wcnt [warps][P]; rpart [kSmallThreads / P][P]; epart [kSmallThreads / epr][epr];
// rprev, total [P]; ecnt [epr]; chv [channels][P] when that fits kNotifyChanBuf.
__host__ __device__ inline SmallSmem small_smem(int P, int E) {
    SmallSmem m;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += (bytes + 15) / 16 * 16;
        return at;
    };
    const int epr = E / P;
    m.wcnt = take(static_cast<size_t>(kSmallWarps) * P * 4);
    m.rpart = take(static_cast<size_t>(kSmallThreads / P) * P * 4);
    m.epart = take(static_cast<size_t>(kSmallThreads / epr) * epr * 4);
    m.rprev = take(static_cast<size_t>(P) * 4);
    m.total = take(static_cast<size_t>(P) * 4);
    m.ecnt = take(static_cast<size_t>(epr) * 4);
    m.chv = take(kNotifyChanBuf * 4);
    m.bytes = o;
    return m;
}

// Grid: P CTAs; CTA s handles source rank s. The warps' token segments are
// the balanced split of T over 32 warps (wq, wr).
template <bool A4>
__global__ void __launch_bounds__(kSmallThreads, 1) notify_small_kernel(const NotifyParams a) {
    pdl_wait_then_release();
    MOE_PROF_BEGIN(kProfNotify);
    extern __shared__ __align__(16) unsigned char smem[];
    const int32_t P = a.P, E = a.E, C = a.C, A = a.A, T = a.T, epr = a.epr;
    const int32_t* __restrict__ ntpr = a.ntpr;
    const int32_t* __restrict__ ntpe = a.ntpe;
    int32_t* __restrict__ rpm = a.rpm;
    int32_t* __restrict__ cpm = a.cpm;
    int32_t* __restrict__ rcpm = a.rcpm;
    int32_t* __restrict__ send_head = a.send_head;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t s = static_cast<int32_t>(blockIdx.x);
    int32_t* wcnt = reinterpret_cast<int32_t*>(smem + a.off_wcnt);
    int32_t* rpart = reinterpret_cast<int32_t*>(smem + a.off_rpart);
    int32_t* epart = reinterpret_cast<int32_t*>(smem + a.off_epart);
    int32_t* rprev = reinterpret_cast<int32_t*>(smem + a.off_rprev);
    int32_t* total = reinterpret_cast<int32_t*>(smem + a.off_total);
    int32_t* ecnt = reinterpret_cast<int32_t*>(smem + a.off_ecnt);
    int32_t* chv = reinterpret_cast<int32_t*>(smem + a.off_chv);

    const int G = (P + 3) >> 2;  // rank groups of 4 (<= 32 here)
    const int lg = a.lg, L = 1 << lg;  // lanes per token: the power of two >= G
    const int tpw = 32 >> lg;
    const int g = lane & (L - 1), tk = lane >> lg;
    const int d = 4 * g;
    const bool gvalid = g < G;
    const int32_t sb = warp * a.wq + min(warp, a.wr);
    const int32_t se = sb + a.wq + (warp < a.wr ? 1 : 0);
    const uint8_t* src_rows = a.itr + static_cast<int64_t>(s) * T * P;

    // --- loads -------------------------------------------------------------
    // rank-prefix partials: column dc over rows rr, rr + R, ... < s
    const int R = a.sR;
    const int rr = div_m(tid, P, a.mP), dc = tid - rr * P;
    int32_t racc = 0;
    if (rr < R)
        for (int32_t q = rr; q < s; q += R) racc += __ldg(ntpr + static_cast<int64_t>(q) * P + dc);
    // expert partials: local expert lc over source ranks qr, qr + Rq, ... < P
    const int Rq = a.sRq;
    const int qr = div_m(tid, epr, a.mE), lc = tid - qr * epr;
    int32_t eacc = 0;
    if (qr < Rq)
        for (int32_t q = qr; q < P; q += Rq) eacc += __ldg(ntpe + static_cast<int64_t>(q) * E + s * epr + lc);
    // this lane's flags, kept for the heads pass
    uint32_t fc[kNotifyCache];
#pragma unroll
    for (int i = 0; i < kNotifyCache; ++i) {
        const int32_t t = sb + tk + i * tpw;
        fc[i] = (gvalid && t < se) ? load_flags<A4>(src_rows + static_cast<int64_t>(t) * P, d, P) : 0u;
    }
    // --- count -------------------------------------------------------------
    int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
#pragma unroll
    for (int i = 0; i < kNotifyCache; ++i) {
        c0 += byte_of(fc[i], 0);
        c1 += byte_of(fc[i], 1);
        c2 += byte_of(fc[i], 2);
        c3 += byte_of(fc[i], 3);
    }
    for (int o = L; o < 32; o <<= 1) {
        c0 += __shfl_xor_sync(0xffffffffu, c0, o);
        c1 += __shfl_xor_sync(0xffffffffu, c1, o);
        c2 += __shfl_xor_sync(0xffffffffu, c2, o);
        c3 += __shfl_xor_sync(0xffffffffu, c3, o);
    }
    if (tk == 0 && gvalid) {
        int32_t* wc = wcnt + warp * P + d;
        wc[0] = c0;
        if (d + 1 < P) wc[1] = c1;
        if (d + 2 < P) wc[2] = c2;
        if (d + 3 < P) wc[3] = c3;
    }
    if (rr < R) rpart[rr * P + dc] = racc;
    if (qr < Rq) epart[qr * epr + lc] = eacc;
    MOE_STAMP(1);
    __syncthreads();
    MOE_STAMP(2);

    // --- reductions, one warp per task --------------------------------------
    const int rows_e = min(Rq, P);
    for (int task = warp; task < 2 * P + epr; task += kSmallWarps) {
        if (task < P) {  // warp offsets of rank task (lane = warp index)
            const int32_t v = lane < kSmallWarps ? wcnt[lane * P + task] : 0;
            const int32_t incl = warp_inclusive_scan(v, lane);
            if (lane < kSmallWarps) wcnt[lane * P + task] = incl - v;
            if (lane == 31) total[task] = incl;
        } else if (task < 2 * P) {  // rank prefix of column task - P
            const int col = task - P;
            int32_t sum = 0;
            for (int r = lane; r < R; r += 32) sum += rpart[r * P + col];
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) rprev[col] = sum;
        } else {  // receive count of local expert task - 2P
            const int l = task - 2 * P;
            int32_t sum = 0;
            for (int r = lane; r < rows_e; r += 32) sum += epart[r * epr + l];
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) ecnt[l] = div_m(sum + A - 1, A, a.mA) * A;  // fits int32 (shape limits)
        }
    }
    __syncthreads();
    MOE_STAMP(3);

    // --- per-rank outputs (from the prefixes and totals alone) -------------
    {
        const int32_t cl = T < C ? (T > 0 ? T - 1 : 0) : C - 1;
        const int32_t cb = T < C ? T : C;
        for (int dd = tid; dd < P; dd += kSmallThreads) {
            const int32_t tot = total[dd], rp = rprev[dd];
            rpm[s * P + dd] = rp + tot;
            for (int32_t c = cl; c < C; ++c) cpm[(static_cast<int64_t>(s) * P + dd) * C + c] = tot;
            for (int32_t c = cb; c < C; ++c) rcpm[(static_cast<int64_t>(dd) * P + s) * C + c] = rp + tot;
            if (s == P - 1) a.nrt[dd] = rp + tot;
        }
    }
    if (warp == kSmallWarps - 1) {  // rank s's receive counts per local expert, scanned
        int32_t carry = 0;
        for (int l0 = 0; l0 < epr; l0 += 32) {
            const int l = l0 + lane;
            const int32_t v = l < epr ? ecnt[l] : 0;
            const int32_t incl = warp_inclusive_scan(v, lane);
            if (l < epr) {
                a.nrtpe[s * epr + l] = v;
                a.reo[s * epr + l] = carry + incl - v;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    if (s == P - 1 && warp == kSmallWarps - 2) {  // packed partition bases
        int64_t run = 0;
        for (int d0 = 0; d0 < P; d0 += 32) {
            const int dd = d0 + lane;
            const int64_t v = dd < P ? static_cast<int64_t>(rprev[dd]) + total[dd] : 0;
            const int64_t incl = warp_inclusive_scan(v, lane);
            if (dd < P) a.part_row_base[dd] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) a.part_row_base[P] = run;
    }

    // --- heads ---------------------------------------------------------------
    const int32_t cq = a.cq, cr = a.cr;
    const int32_t nonempty = min(T, C);  // channels that start before T
    const bool buffered = static_cast<int64_t>(nonempty) * P <= kNotifyChanBuf;
    {
        const int last = (tpw - 1) * L + g;  // lane of this group's last token in a step
        int run[4], rp[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool ok = gvalid && d + j < P;
            run[j] = ok ? wcnt[warp * P + d + j] : 0;
            rp[j] = ok ? rprev[d + j] : 0;
        }
        int32_t nc = sb + tk < se ? next_channel(sb + tk, cq, cr, a.mq1, a.mq0) : C;
        int32_t nb = channel_begin(nc, cq, cr);
#pragma unroll 1
        for (int32_t i = 0, t0 = sb; t0 < se; ++i, t0 += tpw) {
            const int32_t t = t0 + tk;
            const uint32_t f = i == 0 ? fc[0] : (i == 1 ? fc[1] : (i == 2 ? fc[2] : fc[3]));
            const bool tv = gvalid && t < se;
            uint32_t incl = f;
            for (int o = L; o < 32; o <<= 1) {
                const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const uint32_t excl = incl - f;
            const uint32_t step_total = L == 32 ? f : __shfl_sync(0xffffffffu, incl, last);
            if (tv) {
                int loc[4], v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    loc[j] = run[j] + byte_of(excl, j);
                    v[j] = byte_of(f, j) ? rp[j] + loc[j] : -1;
                }
                int32_t* out = send_head + (static_cast<int64_t>(s) * T + t) * P + d;
                if (A4) {
                    *reinterpret_cast<int4*>(out) = make_int4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (d + j < P) out[j] = v[j];
                }
                while (nb < t) nb = channel_begin(++nc, cq, cr);
                if (nb == t) {  // t starts channel nc
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (d + j < P) {
                            if (buffered) {
                                chv[nc * P + d + j] = loc[j];
                            } else {
                                rcpm[(static_cast<int64_t>(d + j) * P + s) * C + nc] = rp[j] + loc[j];
                                if (nc > 0) cpm[(static_cast<int64_t>(s) * P + d + j) * C + nc - 1] = loc[j];
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) run[j] += byte_of(step_total, j);
        }
    }
    MOE_STAMP(4);
    if (buffered) {
        __syncthreads();
        // recv_channel_prefix_matrix[d][s][c] and channel_prefix_matrix[s][d][c-1]
        // for every channel that starts before T, c fastest.
        for (int dd = warp; dd < P; dd += kSmallWarps) {
            int32_t* rrow = rcpm + (static_cast<int64_t>(dd) * P + s) * C;
            int32_t* crow = cpm + (static_cast<int64_t>(s) * P + dd) * C - 1;
            const int32_t rp = rprev[dd];
            for (int c = lane; c < nonempty; c += 32) {
                const int32_t v = chv[c * P + dd];
                rrow[c] = rp + v;
                if (c > 0) crow[c] = v;
            }
        }
    }
    MOE_STAMP(5);
    MOE_STAMP(6);  // stamps 6 and 7 end the kernel, as in the cluster kernel
    MOE_STAMP(7);
    MOE_PROF_END_N(8);
}

struct NotifyPlan {
    bool small;  // one CTA per source rank (notify_small_kernel)
    int cluster;
    int fsteps;  // cluster kernel: flags kept in shared memory (kNotifySmemSteps) or not (0)
    size_t smem;
};

// The cluster kernel keeps a lane's flags in shared memory between its passes
// when one block of rank groups covers P, the register cache does not hold a
// warp's steps and kNotifySmemSteps does.
int notify_fsteps(const moe_shape& s, int cs) {
    const int64_t T = s.S / s.P;
    const int G = (s.P + 3) / 4;
    if (G > 32) return 0;
    int L = 1;
    while (L < G) L <<= 1;
    const int64_t tpw = 32 / L;
    const int64_t seg = ceil_div(T, static_cast<int64_t>(cs) * kNotifyWarps);  // longest warp segment
    const int64_t steps = ceil_div(seg, tpw);
    return (steps > kNotifyCache && steps <= kNotifySmemSteps) ? kNotifySmemSteps : 0;
}

// One CTA of kSmallThreads covers a source rank when each of its kSmallWarps warps
// needs at most kNotifyCache steps (the flags stay in registers) and the rank
// groups fit one warp (P <= 128).
bool notify_small(const moe_shape& s) {
    const int64_t T = s.S / s.P;
    const int G = (s.P + 3) / 4;
    if (G > 32 || s.E / s.P > kSmallThreads) return false;
    int L = 1;
    while (L < G) L <<= 1;
    return T <= static_cast<int64_t>(kSmallWarps) * (32 / L) * kNotifyCache;
}

NotifyPlan notify_plan(const moe_shape& s) {
    const int64_t T = s.S / s.P;
    if (notify_small(s)) {
        NotifyPlan p;
        p.small = true;
        p.cluster = 1;
        p.smem = small_smem(s.P, s.E).bytes;
        return p;
    }
    // Tokens a warp covers per step in the first block of rank groups.
    const int G = (s.P + 3) / 4;
    int L = 1;
    while (L < (G < 32 ? G : 32)) L <<= 1;
    const int64_t tpw = 32 / L;
    // Fewest steps per warp (one if possible), with the grid within about
    // one wave of 4 CTAs per SM; a power of two.
    int c = 1;
    while (c < kNotifyMaxCluster && static_cast<int64_t>(c) * kNotifyWarps * tpw < T) c <<= 1;
    const int64_t wave = 4 * static_cast<int64_t>(device_sm_count());
    while (c > 1 && static_cast<int64_t>(c) * s.P > wave) c >>= 1;
    // the peers' totals and partials (2 x cs x P int32) stay within 64 KB
    while (c > 1 && static_cast<int64_t>(c) * s.P * 8 > 64 * 1024) c >>= 1;
    NotifyPlan p;
    p.small = false;
    p.cluster = c;
    p.fsteps = notify_fsteps(s, c);
    p.smem = notify_smem(s.P, s.E, c, p.fsteps).bytes;
    return p;
}

}  // namespace

MOE_PROFILE_UNIT(notify)

int64_t notify_scratch_bytes(const moe_shape& s) {
    (void)s;
    return 0;
}

cudaError_t launch_notify(const moe_shape& s, const int32_t* ntpr, const int32_t* ntpe,
                          const uint8_t* itr, int32_t* rpm, int32_t* cpm, int32_t* rcpm,
                          int32_t* nrt, int32_t* nrtpe, int32_t* reo, int32_t* send_head,
                          int64_t* part_row_base, void* scratch, cudaStream_t stream) {
    (void)scratch;
    const int64_t T = s.S / s.P;
    const NotifyPlan p = notify_plan(s);
    const bool a4 = (s.P & 3) == 0;
    NotifyParams a{};
    a.P = s.P;
    a.E = s.E;
    a.C = s.num_channels;
    a.A = s.expert_alignment;
    a.epr = s.E / s.P;
    a.T = static_cast<int32_t>(T);
    a.cq = static_cast<int32_t>(T / s.num_channels);
    a.cr = static_cast<int32_t>(T % s.num_channels);
    a.ntpr = ntpr;
    a.ntpe = ntpe;
    a.itr = itr;
    a.rpm = rpm;
    a.cpm = cpm;
    a.rcpm = rcpm;
    a.nrt = nrt;
    a.nrtpe = nrtpe;
    a.reo = reo;
    a.send_head = send_head;
    a.part_row_base = part_row_base;
    a.mq1 = div_magic(a.cq + 1);
    a.mq0 = div_magic(a.cq);
    if (p.small) {
        const void* sfn = a4 ? reinterpret_cast<const void*>(notify_small_kernel<true>)
                             : reinterpret_cast<const void*>(notify_small_kernel<false>);
        cudaError_t e = prepare_kernel(sfn, p.smem, kSmallThreads, nullptr);
        if (e != cudaSuccess) return e;
        a.cs = 1;
        a.wq = static_cast<int32_t>(T / kSmallWarps);
        a.wr = static_cast<int32_t>(T % kSmallWarps);
        const int G = (s.P + 3) / 4;
        a.lg = 0;
        while ((1 << a.lg) < G) ++a.lg;
        a.sR = kSmallThreads / s.P;
        a.sRq = kSmallThreads / a.epr;
        a.mP = div_magic(s.P);
        a.mE = div_magic(a.epr);
        a.mA = div_magic(s.expert_alignment);
        const SmallSmem M = small_smem(s.P, s.E);
        a.off_wcnt = static_cast<int32_t>(M.wcnt);
        a.off_rpart = static_cast<int32_t>(M.rpart);
        a.off_epart = static_cast<int32_t>(M.epart);
        a.off_rprev = static_cast<int32_t>(M.rprev);
        a.off_total = static_cast<int32_t>(M.total);
        a.off_ecnt = static_cast<int32_t>(M.ecnt);
        a.off_chv = static_cast<int32_t>(M.chv);
        return launch_pdl(a4 ? notify_small_kernel<true> : notify_small_kernel<false>, static_cast<unsigned>(s.P),
                          kSmallThreads, p.smem, stream, a);
    }
    const void* fn = a4 ? reinterpret_cast<const void*>(notify_kernel<true>)
                        : reinterpret_cast<const void*>(notify_kernel<false>);
    cudaError_t e = prepare_kernel(fn, p.smem, kNotifyThreads, nullptr);
    if (e != cudaSuccess) return e;
    const int cs = cluster_size_for(fn, p.cluster, kNotifyThreads, p.smem);
    if (cs < 1) return cudaErrorInvalidConfiguration;
    auto kern = a4 ? notify_kernel<true> : notify_kernel<false>;
    a.fsteps = notify_fsteps(s, cs);
    const size_t smem = notify_smem(s.P, s.E, cs, a.fsteps).bytes;  // for the cluster size granted
    if (smem > p.smem) {  // a smaller cluster than planned may need the flag cache
        e = prepare_kernel(fn, smem, kNotifyThreads, nullptr);
        if (e != cudaSuccess) return e;
    }
    a.cs = cs;
    a.lcs = 0;
    while ((1 << a.lcs) < cs) ++a.lcs;
    a.wq = static_cast<int32_t>(T / (cs * kNotifyWarps));
    a.wr = static_cast<int32_t>(T % (cs * kNotifyWarps));
    a.eq = a.epr / cs;
    a.er = a.epr % cs;
    return launch_pdl_cluster(kern, static_cast<unsigned>(s.P) * cs, kNotifyThreads, smem, cs, stream, a);
}

}  // namespace moe
