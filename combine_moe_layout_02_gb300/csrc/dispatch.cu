// dispatch.cu -- the permutation into the ranks' receive partitions (moe_dispatch).
//
// For token g and every rank d with send_head[g][d] >= 0 the slot at row
// part_row_base[d] + send_head[g][d] receives the row (bf16 bits, or int8 +
// fp32 scale) and the triple (source rank, source-local token, lowest k on d):
// "HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 2.3 (slot format) and
// section 3.6 (InputToShare: read the row once, optional dynamic quantisation
// BF16 -> FP32 -> Abs -> ReduceMax -> Scale -> INT8, FillTriple, write out).
// One copy per distinct destination rank: "Ascend DeepEP MoE Dispatch
// Optimization", section "一条 token 如何走完 MoE".
//
// Design (sm_103a). The data path is a pure byte permutation, so it runs on the
// bulk-copy (TMA) engine rather than on the SM's load/store pipes:
//  * Persistent grid, one CTA per token stream (CTA b takes tokens b, b+G, ...).
//  * A ring of `stages` shared-memory row buffers is filled by
//    cp.async.bulk global->shared loads completing on an mbarrier; each source
//    row is read from HBM exactly once.
//  * bf16: for each destination, one lane issues a cp.async.bulk
//    shared->global store of the whole row straight from the ring. Lanes own
//    destinations d = lane, lane+32, ... A ring slot is reused once
//    cp.async.bulk.wait_group.read shows its stores have left shared memory.
//    Warp 0 runs the copies; the other warps write the triples and side arrays
//    for the same tokens in parallel.
//  * int8: a producer warp streams rows into the ring (full / empty
//    mbarriers); consumer warps each take whole tokens: amax by a warp
//    reduction, quantisation (exact round-half-even of x / scale, see
//    quant_one and quant_fast4) into the warp's own int8 row buffer, after
//    which the ring slot goes straight back to the producer; the same bulk
//    stores then fan the int8 row out. One slot per consumer and three
//    consumers per CTA, so several CTAs -- and so many quantising warps --
//    share an SM.
// Every mbarrier wait is bounded; on time-out the CTA records
// MOE_ERR_DEVICE_TIMEOUT, drains its own copies (bounded) and returns.
#include <cuda_bf16.h>

#include "moe_device.cuh"

// Tuning knobs (compile-time): shared-memory budget of the row ring, its
// maximum depth, and how many tokens' bulk-store groups may still be reading
// the ring when a slot is refilled.
#ifndef MOE_DISPATCH_RING_BYTES
#define MOE_DISPATCH_RING_BYTES (96 * 1024)
#endif
#ifndef MOE_DISPATCH_MAX_STAGES
#define MOE_DISPATCH_MAX_STAGES 8
#endif
#ifndef MOE_DISPATCH_STORE_DEPTH
#define MOE_DISPATCH_STORE_DEPTH 1
#endif
// int8 dispatch: ring budget and number of quantising (consumer) warps per CTA.
#ifndef MOE_DISPATCH_INT8_RING_BYTES
#define MOE_DISPATCH_INT8_RING_BYTES (48 * 1024)
#endif
#ifndef MOE_DISPATCH_INT8_CONSUMERS
#define MOE_DISPATCH_INT8_CONSUMERS 3
#endif

namespace moe {
namespace {

constexpr int kBf16Threads = 128;
constexpr int kInt8Consumers = MOE_DISPATCH_INT8_CONSUMERS;
constexpr int kInt8Threads = 32 * (1 + kInt8Consumers);
constexpr int kMaxStages = MOE_DISPATCH_MAX_STAGES;
constexpr int kStoreDepth = MOE_DISPATCH_STORE_DEPTH;
static_assert(kStoreDepth >= 1 && kStoreDepth < kMaxStages, "store depth must leave a free slot");
// The int8 ring has a multiple of kInt8Consumers slots, so a slot's successive
// uses (tokens i and i + stages) belong to the same consumer warp: a warp only
// ever waits on the phase after one it has already consumed, never two phases
// ahead of the barrier.
static_assert(kMaxStages >= kInt8Consumers, "the int8 ring needs a slot per consumer warp");

struct DispatchSmem {
    size_t prb, bars, ring, qbuf, qstride, total;
};

// qbuf: an int8 row buffer for each int8 consumer warp after the ring
// (row_bytes / 2 bytes, rounded up to 128); none for the bf16 kernel.
__host__ __device__ inline DispatchSmem dispatch_smem(int P, int stages, uint32_t row_bytes, bool qbuf = false) {
    DispatchSmem l;
    l.prb = 0;
    l.bars = static_cast<size_t>(round_up(static_cast<int64_t>(P + 1) * 8, 128));
    // full[kMaxStages] then empty[kMaxStages] (the bf16 kernel uses full only)
    l.ring = l.bars + static_cast<size_t>(round_up(2 * kMaxStages * 8, 128));
    l.qbuf = l.ring + static_cast<size_t>(stages) * row_bytes;
    l.qstride = qbuf ? static_cast<size_t>(round_up(row_bytes / 2, 128)) : 0;
    l.total = l.qbuf + static_cast<size_t>(kInt8Consumers) * l.qstride;
    return l;
}

// Routing words of token g a warp needs for its copies and metadata: lane k < K
// holds slot k's expert and weight, lane d < 32 send_head[g][d].
struct TokenRoute {
    int32_t idx, sh0;
    float w;
};

__device__ __forceinline__ TokenRoute load_token_route(const DispatchArgs& a, int64_t g, int lane) {
    TokenRoute r;
    r.idx = lane < a.K ? __ldg(a.topk_idx + g * a.K + lane) : -1;
    r.w = (lane < a.K && a.topk_weights) ? __ldg(a.topk_weights + g * a.K + lane) : 0.f;
    r.sh0 = lane < a.P ? __ldg(a.send_head + g * a.P + lane) : -1;
    return r;
}

// Triple + side arrays for every destination of token g; one warp.
__device__ __forceinline__ void write_token_meta(const DispatchArgs& a, const int64_t* prb, int64_t g, int lane,
                                 TokenRoute rt) {
    const int K = a.K;
    const int32_t idx = rt.idx;
    const float w = rt.w;
    const int32_t dk = (idx >= 0 && idx < a.E) ? idx / a.epr : -1;
    const int32_t src_rank = static_cast<int32_t>(g / a.T);
    const int32_t src_tok = static_cast<int32_t>(g % a.T);
    for (int d0 = 0; d0 < a.P; d0 += 32) {
        const int d = d0 + lane;
        const int32_t sh = d0 == 0 ? rt.sh0 : (d < a.P ? __ldg(a.send_head + g * a.P + d) : -1);
        uint32_t todo = __ballot_sync(0xffffffffu, sh >= 0);
        while (todo) {
            const int j = __ffs(todo) - 1;
            todo &= todo - 1;
            const int dd = d0 + j;
            const int32_t shd = __shfl_sync(0xffffffffu, sh, j);
            const int64_t lo = prb[dd], hi = prb[dd + 1];
            const int64_t row = lo + shd;
            if (shd >= hi - lo || row < 0 || row >= a.arena_rows) continue;  // reported by the copy path
            const bool on = dk == dd;
            const uint32_t kb = __ballot_sync(0xffffffffu, on);
            if (lane < K) {
                if (a.recv_topk_idx) a.recv_topk_idx[row * K + lane] = on ? idx % a.epr : -1;
                if (a.recv_topk_weights) a.recv_topk_weights[row * K + lane] = on ? w : 0.f;
            }
            if (lane == 0) {
                if (a.recv_src_idx) a.recv_src_idx[row] = src_tok;
                // The triple fills its whole 32-byte sector (zero padded) so the
                // sector never needs a read-modify-write on its way to DRAM.
                int4* t = reinterpret_cast<int4*>(a.arena + row * a.stride + a.triple_off);
                t[0] = make_int4(src_rank, src_tok, kb ? __ffs(kb) - 1 : -1, 0);
                t[1] = make_int4(0, 0, 0, 0);
            }
        }
    }
}

// Row address of destination d for token g, or nullptr (and an error) when the
// row is outside its partition or the arena.
__device__ __forceinline__ uint8_t* slot_of(const DispatchArgs& a, const int64_t* prb, int d, int32_t sh) {
    const int64_t lo = prb[d], hi = prb[d + 1];
    const int64_t row = lo + sh;
    if (sh < hi - lo && row >= 0 && row < a.arena_rows) return a.arena + row * a.stride;
    raise_error(a.err, MOE_ERR_CAPACITY);
    return nullptr;
}

// Expert-major layout: destination row of slot (g, lane), or nullptr. Lanes
// k < K carry slot k; the row is part_row_base[d] + slot_row[g][k].
__device__ __forceinline__ uint8_t* expert_slot_of(const DispatchArgs& a, const int64_t* prb, int64_t g,
                                                   int lane, int64_t* row_out) {
    if (lane >= a.K) return nullptr;
    const int32_t e = __ldg(a.topk_idx + g * a.K + lane);
    const int32_t sr = __ldg(a.slot_row + g * a.K + lane);
    if (e < 0 || e >= a.E || sr < 0) return nullptr;
    const int d = e / a.epr;
    uint8_t* dst = slot_of(a, prb, d, sr);
    if (dst) *row_out = prb[d] + sr;
    return dst;
}

// Expert-major layout: triple (source rank, source-local token, k) and side
// arrays of each slot of token g; lane k writes slot k's.
__device__ void write_slot_meta(const DispatchArgs& a, const int64_t* prb, int64_t g, int lane) {
    if (lane >= a.K) return;
    const int32_t e = __ldg(a.topk_idx + g * a.K + lane);
    const int32_t sr = __ldg(a.slot_row + g * a.K + lane);
    if (e < 0 || e >= a.E || sr < 0) return;
    const int d = e / a.epr;
    const int64_t lo = prb[d], hi = prb[d + 1], row = lo + sr;
    if (sr >= hi - lo || row < 0 || row >= a.arena_rows) return;  // reported by the copy path
    const int32_t t = static_cast<int32_t>(g % a.T);
    int4* trip = reinterpret_cast<int4*>(a.arena + row * a.stride + a.triple_off);
    trip[0] = make_int4(static_cast<int32_t>(g / a.T), t, lane, 0);
    trip[1] = make_int4(0, 0, 0, 0);
    if (a.recv_src_idx) a.recv_src_idx[row] = t;
    if (a.recv_weight) a.recv_weight[row] = a.topk_weights ? __ldg(a.topk_weights + g * a.K + lane) : 1.f;
}

__device__ void load_prb_and_init(const DispatchArgs& a, int64_t* prb, uint64_t* bars) {
    for (int i = threadIdx.x; i <= a.P; i += blockDim.x) prb[i] = a.part_row_base[i];
    if (threadIdx.x == 0) {
        for (int st = 0; st < a.stages; ++st) mbar_init(&bars[st], 1);
        mbar_init_fence();
    }
    __syncthreads();
}

// After a failed wait: wait (bounded) for the loads this CTA still has in flight
// into its ring, so that no copy lands in shared memory after the CTA exits.
__device__ void drain_loads(uint64_t* bars, int stages, int64_t first, int64_t last_issued) {
    for (int64_t j = first; j <= last_issued; ++j) mbar_wait(&bars[j % stages], (j / stages) & 1);
}

template <bool EXPERT>
__global__ void __launch_bounds__(kBf16Threads) dispatch_bf16_kernel(const DispatchArgs a) {
    pdl_wait_then_release();
    MOE_PROF_BEGIN(kProfDispatch);
    extern __shared__ __align__(128) unsigned char smem[];
    const DispatchSmem L = dispatch_smem(a.P, a.stages, a.row_bytes);
    int64_t* prb = reinterpret_cast<int64_t*>(smem + L.prb);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    unsigned char* ring = smem + L.ring;
    load_prb_and_init(a, prb, bars);
    MOE_STAMP(1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int64_t G = gridDim.x;
    const int64_t n_local = blockIdx.x < a.S ? (a.S - 1 - blockIdx.x) / G + 1 : 0;

    if (warp != 0) {
        for (int64_t i = warp - 1; i < n_local; i += nwarps - 1) {
            if constexpr (EXPERT) {
                write_slot_meta(a, prb, blockIdx.x + i * G, lane);
            } else {
                const int64_t g = blockIdx.x + i * G;
                write_token_meta(a, prb, g, lane, load_token_route(a, g, lane));
            }
        }
        return;
    }

    const int NS = a.stages;
    const uint32_t RB = a.row_bytes;
    int64_t last_issued = -1;
    if (lane == 0) {
        const int64_t npro = n_local < NS ? n_local : NS;
        for (int64_t i = 0; i < npro; ++i) {
            mbar_arrive_expect_tx(&bars[i], RB);
            bulk_load(ring + i * RB, a.x + (blockIdx.x + i * G) * a.H, RB, &bars[i]);
        }
        last_issued = npro - 1;
    }
    __syncwarp();
    bool failed = false;
    int64_t i = 0;
    for (; i < n_local; ++i) {
        const int slot = static_cast<int>(i % NS);
        const int64_t g = blockIdx.x + i * G;
        int32_t sh0 = -1;
        uint8_t* xdst = nullptr;
        if constexpr (EXPERT) {
            int64_t row;
            xdst = expert_slot_of(a, prb, g, lane, &row);
        } else {
            sh0 = lane < a.P ? __ldg(a.send_head + g * a.P + lane) : -1;
        }
        const bool ok = mbar_wait(&bars[slot], static_cast<uint32_t>((i / NS) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            failed = true;
            break;
        }
        const unsigned char* src = ring + static_cast<size_t>(slot) * RB;
        if constexpr (EXPERT) {
            if (xdst) bulk_store(xdst, src, RB);
        } else {
            for (int d0 = 0; d0 < a.P; d0 += 32) {
                const int d = d0 + lane;
                const int32_t sh = d0 == 0 ? sh0 : (d < a.P ? __ldg(a.send_head + g * a.P + d) : -1);
                if (sh >= 0) {
                    uint8_t* dst = slot_of(a, prb, d, sh);
                    if (dst) bulk_store(dst, src, RB);
                }
            }
        }
        bulk_commit();
        // Token i-D's stores have left its slot once at most D groups (tokens
        // i-D+1 .. i) still read shared memory; refill that slot.
        bulk_wait_read<kStoreDepth>();
        __syncwarp();
        if (lane == 0 && i >= kStoreDepth) {
            const int64_t nxt = i - kStoreDepth + NS;
            if (nxt < n_local) {
                const int ps = static_cast<int>((i - kStoreDepth) % NS);
                mbar_arrive_expect_tx(&bars[ps], RB);
                bulk_load(ring + static_cast<size_t>(ps) * RB, a.x + (blockIdx.x + nxt * G) * a.H, RB,
                          &bars[ps]);
                last_issued = nxt;
            }
        }
        __syncwarp();
    }
    MOE_STAMP(2);
    bulk_wait<0>();
    MOE_STAMP(3);
    if (failed && lane == 0) {
        raise_error(a.err, MOE_ERR_DEVICE_TIMEOUT);
        drain_loads(bars, NS, i, last_issued);
    }
    MOE_PROF_END_N(4);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// q = rint(x / scale) with round-half-even, exactly as with IEEE division, for
// finite x. Bound on the quotient: scale = amax / 127 rounded, with an error
// of at most half an ulp -- relative 2^-24 for a normal scale, absolute 2^-150
// for a subnormal one. A bf16 amax is at least 2^-133 (the smallest bf16
// denormal), so scale >= amax / 127 - 127 * 2^-17 * (amax / 127) and
// |x / scale| <= amax / scale <= 127 / (1 - 127 * 2^-17) < 127.13 < 127.5:
// q is already in [-127, 127], and the clamp the definition states never acts.
// The quotient is taken as t = x * r, r = 1 / scale rounded (two roundings of
// relative 2^-24 each): |t - x / scale| <= 127.13 * 2^-23 < 2^-15, so rounding
// t gives the same integer unless t lies within 2^-15 of a half-integer; only
// then (or when r is not finite) is the division done.
__device__ __forceinline__ int32_t quant_one(float x, float scale, float r, bool fast) {
    const float t = __fmul_rn(x, r);
    int32_t q = __float2int_rn(t);
    if (!(fast && fabsf(t - __int2float_rn(q)) < 0.5f - 0x1p-15f)) q = __float2int_rn(__fdiv_rn(x, scale));
    return q;
}

// Adding 1.5 * 2^23 to a binary32 |t| < 2^22 rounds it to an integer, half to
// even (IEEE round to nearest); the sum's low byte is then that integer mod 256.
constexpr float kRoundMagic = 12582912.0f;

// Packed binary32 pairs (two independent IEEE round-to-nearest operations per
// instruction): the low word holds one element, the high word the next.
__device__ __forceinline__ uint64_t f32x2_pack(uint32_t lo, uint32_t hi) {
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float f32x2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f32x2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// 4 bf16 (two words) -> 4 int8 bytes of rint(x * r), with no conversion
// instructions, two elements per arithmetic instruction. `near` is set when
// some t = x * r lies within 2^-15 of a half-integer, where rounding t may
// differ from rounding x / scale (see quant_one); the caller then redoes the
// chunk with division.
__device__ __forceinline__ uint32_t quant_fast4(uint32_t w0, uint32_t w1, float r, bool& near) {
    const uint64_t rr = f32x2_pack(__float_as_uint(r), __float_as_uint(r));
    const uint64_t mm = f32x2_pack(__float_as_uint(kRoundMagic), __float_as_uint(kRoundMagic));
    const uint64_t t0 = f32x2_mul(f32x2_pack(w0 << 16, w0 & 0xffff0000u), rr);
    const uint64_t t1 = f32x2_mul(f32x2_pack(w1 << 16, w1 & 0xffff0000u), rr);
    const uint64_t u0 = f32x2_add(t0, mm), u1 = f32x2_add(t1, mm);
    const uint64_t d0 = f32x2_sub(t0, f32x2_sub(u0, mm)), d1 = f32x2_sub(t1, f32x2_sub(u1, mm));
    const float m = fmaxf(fmaxf(fabsf(f32x2_lo(d0)), fabsf(f32x2_hi(d0))),
                          fmaxf(fabsf(f32x2_lo(d1)), fabsf(f32x2_hi(d1))));
    near |= m >= 0.5f - 0x1p-15f;
    const uint32_t lo = __byte_perm(static_cast<uint32_t>(u0), static_cast<uint32_t>(u0 >> 32), 0x0040);
    const uint32_t hi = __byte_perm(static_cast<uint32_t>(u1), static_cast<uint32_t>(u1 >> 32), 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// 8 bf16 (one 16-byte chunk) -> 8 int8, packed little-endian.
__device__ __forceinline__ uint2 quant_chunk(uint4 v, float scale, float r, bool fast, bool zero) {
    if (zero) return make_uint2(0u, 0u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int32_t q0 = quant_one(bf16_lo(w[2 * h]), scale, r, fast);
        const int32_t q1 = quant_one(bf16_hi(w[2 * h]), scale, r, fast);
        const int32_t q2 = quant_one(bf16_lo(w[2 * h + 1]), scale, r, fast);
        const int32_t q3 = quant_one(bf16_hi(w[2 * h + 1]), scale, r, fast);
        const uint32_t lo = __byte_perm(static_cast<uint32_t>(q0), static_cast<uint32_t>(q1), 0x0040);
        const uint32_t hi = __byte_perm(static_cast<uint32_t>(q2), static_cast<uint32_t>(q3), 0x0040);
        o[h] = __byte_perm(lo, hi, 0x5410);
    }
    return make_uint2(o[0], o[1]);
}

// The divisions of the int8 path (once per token, and per chunk only near a
// half-integer) are out-of-line calls, so the registers of the hot loop are
// not saved around them on every token.
__device__ __noinline__ float scale_of_amax(float m) { return __fdiv_rn(m, 127.0f); }
__device__ __noinline__ uint2 quant_chunk_exact(uint4 v, float scale, bool zero) {
    return quant_chunk(v, scale, 0.f, false, zero);
}

// max |x| over 8 bf16, as a bf16 pair (bf16 max is exact).
__device__ __forceinline__ __nv_bfloat162 absmax_chunk(__nv_bfloat162 m, uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b;
        memcpy(&b, &w[i], 4);
        m = __hmax2(m, __habs2(b));
    }
    return m;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// int8 dispatch. Warp 0 is the producer: it streams source rows into the ring
// (bulk loads completing on full[slot]) and reuses a slot once the consumer
// that read it arrives on empty[slot]. Warps 1..kInt8Consumers each take
// whole tokens in turn: amax by a warp reduction, scale = amax / 127, the
// quantised row written to the warp's own int8 row buffer, the slot handed
// back to the producer, then one bulk store per destination from the row
// buffer, the scale block and the triple / side arrays. The next row's load
// thus overlaps this row's stores; the row buffer is rewritten once those
// stores have read it. No block-wide barrier on the token path.
template <bool EXPERT>
__global__ void __launch_bounds__(kInt8Threads) dispatch_int8_kernel(const DispatchArgs a) {
    // Waits for the previous kernel but does not let the next one be scheduled
    // early: with many small CTAs per SM here, the next kernel's CTAs resident
    // beside these slowed the pair down (measured: dispatch + combine 835 vs
    // 761 us at P=8, H=7168). The next kernel launches as these CTAs exit.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    MOE_PROF_BEGIN(kProfDispatchInt8);
    extern __shared__ __align__(128) unsigned char smem[];
    const DispatchSmem L = dispatch_smem(a.P, a.stages, a.row_bytes, true);
    int64_t* prb = reinterpret_cast<int64_t*>(smem + L.prb);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kMaxStages;
    unsigned char* ring = smem + L.ring;
    for (int i = threadIdx.x; i <= a.P; i += blockDim.x) prb[i] = a.part_row_base[i];
    if (threadIdx.x == 0) {
        for (int st = 0; st < a.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], 1);
        }
        mbar_init_fence();
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t n_local = blockIdx.x < a.S ? (a.S - 1 - blockIdx.x) / G + 1 : 0;
    const int NS = a.stages;
    const uint32_t RB = a.row_bytes;

    if (warp == 0) {
        if (lane != 0) return;
        int64_t issued = 0;
        bool failed = false;
        for (; issued < n_local; ++issued) {
            const int slot = static_cast<int>(issued % NS);
            if (issued >= NS && !mbar_wait(&empty[slot], static_cast<uint32_t>(((issued / NS) - 1) & 1))) {
                failed = true;
                break;
            }
            mbar_arrive_expect_tx(&full[slot], RB);
            bulk_load(ring + static_cast<size_t>(slot) * RB, a.x + (blockIdx.x + issued * G) * a.H, RB,
                      &full[slot]);
        }
        if (failed) raise_error(a.err, MOE_ERR_DEVICE_TIMEOUT);
        // Loads still in flight land before the CTA may exit.
        const int64_t first = issued > NS ? issued - NS : 0;
        drain_loads(full, NS, first, issued - 1);
        MOE_PROF_END_N(1);
        return;
    }

    const int cw = warp - 1;
    const int nchunks = a.H / 8;
    unsigned char* q = smem + L.qbuf + static_cast<size_t>(cw) * L.qstride;  // this warp's int8 row
    // Profile build: consumer 0's cycles per step, summed over its tokens.
    long long pw = 0, pa = 0, pq = 0, ps = 0, pn = 0;
    (void)pw, (void)pa, (void)pq, (void)ps, (void)pn;
    for (int64_t i = cw; i < n_local; i += kInt8Consumers) {
        const int slot = static_cast<int>(i % NS);
        const int64_t g = blockIdx.x + i * G;
        long long c_ = MOE_PROF_CLOCK();
        const bool ok = mbar_wait(&full[slot], static_cast<uint32_t>((i / NS) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) raise_error(a.err, MOE_ERR_DEVICE_TIMEOUT);
            break;
        }
        {
            const long long c1 = MOE_PROF_CLOCK();
            pw += c1 - c_;
            c_ = c1;
        }
        const uint4* row = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * RB);
        __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll 4
        for (int j = lane; j < nchunks; j += 32) m2 = absmax_chunk(m2, row[j]);
        float m = fmaxf(__bfloat162float(m2.x), __bfloat162float(m2.y));
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float scale = scale_of_amax(m);
        const bool zero = m == 0.f;
        {
            const long long c1 = MOE_PROF_CLOCK();
            pa += c1 - c_;
            c_ = c1;
        }
        const float r = zero ? 0.f : __frcp_rn(scale);
        const bool fast = !zero && isfinite(r);
        // The previous token's stores have read the row buffer.
        bulk_wait_read<0>();
        __syncwarp();
        for (int j0 = 0; j0 < nchunks; j0 += 32) {
            const int j = j0 + lane;
            if (j < nchunks) {
                const uint4 v = row[j];
                uint2 o;
                if (fast) {
                    bool near = false;
                    o.x = quant_fast4(v.x, v.y, r, near);
                    o.y = quant_fast4(v.z, v.w, r, near);
                    if (near) o = quant_chunk_exact(v, scale, false);
                } else {
                    o = quant_chunk_exact(v, scale, zero);
                }
                reinterpret_cast<uint2*>(q)[j] = o;
            }
        }
        // Every lane has read the bf16 row: the slot goes back to the producer
        // now, so the next load overlaps this token's stores.
        __syncwarp();
        {
            const long long c1 = MOE_PROF_CLOCK();
            pq += c1 - c_;
            c_ = c1;
        }
        if (lane == 0) mbar_arrive(&empty[slot]);
        fence_proxy_async_smem();
        __syncwarp();
        const int nfan = EXPERT ? a.K : a.P;
        for (int d = lane; d < nfan; d += 32) {
            uint8_t* dst = nullptr;
            if constexpr (EXPERT) {
                int64_t rowi;
                dst = expert_slot_of(a, prb, g, d, &rowi);
            } else {
                const int32_t sh = __ldg(a.send_head + g * a.P + d);
                if (sh >= 0) dst = slot_of(a, prb, d, sh);
            }
            if (dst) {
                bulk_store(dst, q, static_cast<uint32_t>(a.H));
                // Scale plus zero padding: one whole 32-byte sector.
                int4* sc = reinterpret_cast<int4*>(dst + a.scale_off);
                sc[0] = make_int4(__float_as_int(scale), 0, 0, 0);
                sc[1] = make_int4(0, 0, 0, 0);
            }
        }
        bulk_commit();
        if constexpr (EXPERT)
            write_slot_meta(a, prb, g, lane);
        else
            write_token_meta(a, prb, g, lane, load_token_route(a, g, lane));
        ps += MOE_PROF_CLOCK() - c_;
        ++pn;
    }
    bulk_wait<0>();
    if (cw == 0 && lane == 0) {
        // slots: 1 wait for the row, 2 amax, 3 quantisation, 4 stores and
        // metadata (cycles summed over the tokens), 5 tokens
        MOE_PROF_PUT(1, pw);
        MOE_PROF_PUT(2, pa);
        MOE_PROF_PUT(3, pq);
        MOE_PROF_PUT(4, ps);
        MOE_PROF_PUT(5, pn);
    }
}

}  // namespace

template <bool EXPERT>
cudaError_t launch_dispatch_mode(const moe_shape& s, DispatchArgs a, cudaStream_t stream) {
    if (a.S == 0) return cudaSuccess;
    const bool quant = s.quant != 0;
    // Ring depth: as many rows as fit in the ring budget, at least one more
    // than the store depth (and 2), at most kMaxStages.
    int stages;
    if (quant) {
        // A multiple of the consumer count (see kInt8Consumers), at least one
        // slot per consumer, at most kMaxStages.
        const int per = static_cast<int>(MOE_DISPATCH_INT8_RING_BYTES / (a.row_bytes * kInt8Consumers));
        const int groups_max = kMaxStages / kInt8Consumers;
        stages = kInt8Consumers * (per < 1 ? 1 : (per > groups_max ? groups_max : per));
    } else {
        stages = static_cast<int>(MOE_DISPATCH_RING_BYTES / a.row_bytes);
        const int min_stages = kStoreDepth + 1 > 2 ? kStoreDepth + 1 : 2;
        stages = stages < min_stages ? min_stages : (stages > kMaxStages ? kMaxStages : stages);
    }
    a.stages = stages;
    const DispatchSmem L = dispatch_smem(s.P, stages, a.row_bytes, quant);
    if (L.total > static_cast<size_t>(device_optin_smem())) return cudaErrorInvalidConfiguration;
    const void* fn = quant ? reinterpret_cast<const void*>(dispatch_int8_kernel<EXPERT>)
                           : reinterpret_cast<const void*>(dispatch_bf16_kernel<EXPERT>);
    const int threads = quant ? kInt8Threads : kBf16Threads;
    int per_sm = 0;
    cudaError_t e = prepare_kernel(fn, L.total, threads, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
    if (grid > a.S) grid = a.S;
    if (quant)
        return launch_pdl(dispatch_int8_kernel<EXPERT>, static_cast<unsigned>(grid), threads, L.total, stream, a);
    return launch_pdl(dispatch_bf16_kernel<EXPERT>, static_cast<unsigned>(grid), threads, L.total, stream, a);
}

cudaError_t launch_dispatch(const moe_shape& s, DispatchArgs a, cudaStream_t stream) {
    return launch_dispatch_mode<false>(s, a, stream);
}

cudaError_t launch_dispatch_expert(const moe_shape& s, DispatchArgs a, cudaStream_t stream) {
    return launch_dispatch_mode<true>(s, a, stream);
}

MOE_PROFILE_UNIT(dispatch)

}  // namespace moe
