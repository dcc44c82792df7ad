// rc_bf16.cu -- the same path with a 16-bit ring (RC_F_BF16_CACHE): the non-FP8
// cache of the comparison the cpdf.ai blog draws in "Blackwell, escalabilidade
// e limites do decodificador" (the FP8 cache saved 17.0 ms a step on H100 and
// cost 2.4-6.7 ms on B200, whose build had no per-head-scaled FP8 attention).
// Keys are still rotated once, at write time, and re-rotated on a position
// reset; only the storage differs: keys rounded once to bf16 instead of
// per-head E4M3, values kept at 16 bits instead of E4M3.
//
// The values are stored as fp16, converted once at write time from the bf16
// input (exact for 2^-17 <= |v| < 65520 and for zero; smaller magnitudes round
// to fp16's subnormal step, larger ones become +-inf).  P.V runs on fp16
// because P needs fp16's 11 bits; converting V at write time, as the ring does
// with RoPE, spares every attention call the conversion and its shared-memory
// traffic, and gives the same attention result as converting at read time.
//
// KB1 bf16_write_kernel: K rotated by RoPE (fp32, fp64-angle cos/sin) and
//    rounded once to bf16 into the K tile; V converted to fp16 into the
//    transposed Vt tile through a shared-memory transpose.
// KB2 bf16_rotate_kernel: every stored key of every layer re-rotated by the
//    delta and rounded to bf16 again, in place (no scales to recompute).
// KB3 bf16_attn_kernel: one CTA = one head x 128 query rows.  The queries are
//    rotated and split into two bf16 pieces (hi + lo, ~16 significant bits)
//    held in TMEM; S = Q K^T on tcgen05 kind::f16 with Q from TMEM and K from
//    shared memory (two MMAs per K step), P in fp16, O += P V on kind::f16
//    with the fp16 Vt tile as it lands.  The scores are double-buffered in
//    TMEM over KV tiles: Q.K of tile j + 2 is queued behind P.V of tile j, so
//    the tensor pipe works while the softmax processes the next tile; K and
//    V tiles are triple-buffered.  Warps: 0 loader (K and V tiles by bulk
//    copy), 1 MMA issuer, 2..5 softmax (one TMEM lane quadrant each), 6
//    checker (certifies the next step's K and V tiles); all eight prepare
//    the queries.
#include <atomic>

#include "rc_device.cuh"
#include "rc_internal.h"
#include "rc_layout.h"

namespace rc {

// ---------------------------------------------------------------- KB1 write

constexpr int kBWriteTokens = 64;  // tokens per CTA
constexpr int kBWriteThreads = 256;

template <int D>
__global__ void __launch_bounds__(kBWriteThreads) bf16_write_kernel(WriteParams p) {
    constexpr int EPL = D / 32;  // dims per lane of a row
    __shared__ __align__(16) __half vs[kBWriteTokens][D + 8];
    __shared__ int s_slot[kBWriteTokens];
    const int h = blockIdx.y;
    const int t0 = blockIdx.x * kBWriteTokens;
    const int cnt = min(kBWriteTokens, p.n - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dim0 = lane * EPL;
    auto slot_of = [&](int t) -> int {
        if (p.pos == nullptr) {
            const int s = p.slot0 + t;  // t < n <= C
            return s >= p.C ? s - p.C : s;
        }
        return static_cast<int>(floormod64(p.pos[t] - p.delta_total, p.C));
    };
    // K: a warp per token row; RoPE in fp32 (the write path's rounding order),
    // one bf16 rounding, EPL consecutive dims (2 EPL bytes) per lane into the tile
    for (int tl = warp; tl < cnt; tl += kBWriteThreads / 32) {
        const int t = t0 + tl;
        const int slot = slot_of(t);
        if (lane == 0) s_slot[tl] = slot;
        const size_t src = (static_cast<size_t>(t) * p.H + h) * D + dim0;
        __nv_bfloat16 kb[EPL], vb[EPL];
        if constexpr (EPL == 4) {
            *reinterpret_cast<uint2*>(kb) = *reinterpret_cast<const uint2*>(p.K + src);
            *reinterpret_cast<uint2*>(vb) = *reinterpret_cast<const uint2*>(p.V + src);
        } else {
            *reinterpret_cast<uint32_t*>(kb) = *reinterpret_cast<const uint32_t*>(p.K + src);
            *reinterpret_cast<uint32_t*>(vb) = *reinterpret_cast<const uint32_t*>(p.V + src);
        }
        __nv_bfloat16 ko[EPL];
#pragma unroll
        for (int j = 0; j < EPL / 2; ++j) {
            const float2 cs = p.rope[static_cast<size_t>(t) * (D / 2) + dim0 / 2 + j];
            float x, y;
            rotate_pair(__bfloat162float(kb[2 * j]), __bfloat162float(kb[2 * j + 1]), cs.x, cs.y, x, y);
            ko[2 * j] = __float2bfloat16_rn(x);
            ko[2 * j + 1] = __float2bfloat16_rn(y);
        }
        uint8_t* kt = p.kc + (static_cast<size_t>(h) * p.T + (slot >> 7)) * (kTileSlots * D * 2) +
                      bktile_off(slot & 127, dim0);
        if constexpr (EPL == 4)
            *reinterpret_cast<uint2*>(kt) = *reinterpret_cast<const uint2*>(ko);
        else
            *reinterpret_cast<uint32_t*>(kt) = *reinterpret_cast<const uint32_t*>(ko);
#pragma unroll
        for (int e = 0; e < EPL; ++e) vs[tl][dim0 + e] = __float2half_rn(__bfloat162float(vb[e]));
        if (lane == 0 && h == 0) p.grp[slot] = p.group;
    }
    __syncthreads();
    // V transposed: a warp per dim row, the lanes over the tokens, so each store
    // instruction writes the consecutive slots of one dim row
    uint8_t* vhead = p.vt + static_cast<size_t>(h) * p.T * (kTileSlots * D * 2);
    for (int d = warp; d < D; d += kBWriteThreads / 32) {
        for (int tl = lane; tl < cnt; tl += 32) {
            const int slot = s_slot[tl];
            *reinterpret_cast<__half*>(vhead + static_cast<size_t>(slot >> 7) * (kTileSlots * D * 2) +
                                       bvtile_off(d, slot & 127, D)) = vs[tl][d];
        }
    }
}

cudaError_t launch_bf16_write(const WriteParams& p, int D, cudaStream_t s) {
    dim3 grid((p.n + kBWriteTokens - 1) / kBWriteTokens, p.H);
    if (D == 128)
        bf16_write_kernel<128><<<grid, kBWriteThreads, 0, s>>>(p);
    else
        bf16_write_kernel<64><<<grid, kBWriteThreads, 0, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- KB2 rotate

constexpr int kBRotThreads = 256;

// One CTA per (tile, head, layer); a thread per 16-byte chunk (8 dims = 4
// pairs) of a row, rows of empty slots skipped.
template <int D>
__global__ void __launch_bounds__(kBRotThreads) bf16_rotate_kernel(RotateParams p) {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    __shared__ float2 s_cs[kMaxHalfDim];
    if (threadIdx.x < D / 2) s_cs[threadIdx.x] = p.cs[threadIdx.x];
    __syncthreads();
    const int tile = blockIdx.x, h = blockIdx.y, l = blockIdx.z;
    uint8_t* kt = p.kc + ((static_cast<size_t>(l) * p.H + h) * p.T + tile) * (kTileSlots * D * 2);
    const int32_t* grp = p.grp + static_cast<size_t>(l) * p.Cpad + tile * kTileSlots;
    for (int u = threadIdx.x; u < kTileSlots * CPR; u += kBRotThreads) {
        const int row = u / CPR, c = u - row * CPR;  // physical chunk c of the row
        if (grp[row] < 0) continue;
        const int blk = c >> 3, pc = c & 7;
        const int dim0 = blk * 64 + ((pc ^ (row & 7)) << 3);  // logical dims of the chunk
        uint8_t* at = kt + blk * (kTileSlots * 128) + row * 128 + (pc << 4);
        uint4 w = *reinterpret_cast<const uint4*>(at);
        uint32_t* wv = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 ab = *reinterpret_cast<const __nv_bfloat162*>(&wv[j]);
            const float2 cs = s_cs[dim0 / 2 + j];
            float x, y;
            rotate_pair(__low2float(ab), __high2float(ab), cs.x, cs.y, x, y);
            const __nv_bfloat162 o = __floats2bfloat162_rn(x, y);
            wv[j] = *reinterpret_cast<const uint32_t*>(&o);
        }
        *reinterpret_cast<uint4*>(at) = w;
    }
}

cudaError_t launch_bf16_rotate(const RotateParams& p, int D, int layers, cudaStream_t s) {
    dim3 grid(p.T, p.H, layers);
    if (D == 128)
        bf16_rotate_kernel<128><<<grid, kBRotThreads, 0, s>>>(p);
    else
        bf16_rotate_kernel<64><<<grid, kBRotThreads, 0, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- KB3 attention

constexpr int kBAttnWarps = 8;
constexpr int kBAttnThreads = kBAttnWarps * 32;
constexpr int kBRows = 128;                        // query rows (one M tile) per CTA
constexpr int kBStages = 3;                        // K tiles and V buffers in flight
constexpr int kBWarpLoad = 0, kBWarpMma = 1, kBWarpSm0 = 2, kBWarpSmEnd = 6, kBWarpCheck = 6;
constexpr int kBNbP = 1;                           // named barrier: P, V and the next K of a tile are ready
constexpr int kBNbPThreads = 4 * 32 + 32 + 32;     // softmax warps, MMA warp, checker warp

enum : int {
    BB_K_FULL = 0,                    // [3] K tile (and, on a masked ring, its write groups) landed
    BB_K_EMPTY = BB_K_FULL + 3,       // [3] its Q.K finished (and on a masked ring the softmax read the groups)
    BB_V_FULL = BB_K_EMPTY + 3,       // [3] fp16 Vt tile landed
    BB_V_EMPTY = BB_V_FULL + 3,       // [3] its P.V finished (also: O holds that P.V, for an O rescale)
    BB_S_FULL = BB_V_EMPTY + 3,       // [2] scores of a tile in TMEM score buffer b
    BB_O_DONE = BB_S_FULL + 2,
    BB_DRAIN = BB_O_DONE + 1,
    BB_COUNT = BB_DRAIN + 1
};

template <int D>
struct BAttnLayout {
    static constexpr uint32_t kTile = kTileSlots * D * 2;   // bytes of a bf16 K or Vt tile
    static constexpr uint32_t kK = 0;                        // [3] K tiles
    static constexpr uint32_t kV = kK + kBStages * kTile;    // [3] fp16 Vt tiles
    static constexpr uint32_t kGrp = kV + kBStages * kTile;  // [3][128] int32 write groups (masked rings)
    static constexpr uint32_t kBar = kGrp + kBStages * kTileSlots * 4;
    static constexpr uint32_t kMisc = kBar + 8 * BB_COUNT;
    static constexpr uint32_t kTotal = kMisc + 64;
    static constexpr uint32_t kAlloc = kTotal + 1024;
};

// TMEM columns: scores S0 | S1 | O | Q hi | Q lo
constexpr uint32_t kBColS = 0, kBColO = 256, kBColQ = 384;

template <int D>
__global__ void __launch_bounds__(kBAttnThreads, 1) bf16_attn_kernel(AttnParams p) {
    using Lay = BAttnLayout<D>;
    constexpr uint32_t kBlk = kTileSlots * 128;  // bytes of one 64-element block of 128 rows
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);  // [0] tmem, [2] abort
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int row0 = blockIdx.x * kBRows;
    const int T = p.T;
    AbortState ab{reinterpret_cast<volatile uint32_t*>(&misc[2]), p.status, p.wait_ns};

    if (tid == 0) {
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&bars[BB_K_FULL + s], 1);
            mbar_init(&bars[BB_K_EMPTY + s], p.masked ? 1 + 4 : 1);
            mbar_init(&bars[BB_V_FULL + s], 1);
            mbar_init(&bars[BB_V_EMPTY + s], 1);
        }
        for (int b = 0; b < 2; ++b) mbar_init(&bars[BB_S_FULL + b], 1);
        mbar_init(&bars[BB_O_DONE], 1);
        mbar_init(&bars[BB_DRAIN], 1);
        misc[2] = 0u;
        fence_mbar_init();
    }
    if (warp == kBWarpMma) {
        tmem_alloc(&misc[0], 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    auto k_ptr = [&](int s) { return smem + Lay::kK + s * Lay::kTile; };
    auto v_ptr = [&](int s) { return smem + Lay::kV + s * Lay::kTile; };
    auto grp_ptr = [&](int s) { return reinterpret_cast<int32_t*>(smem + Lay::kGrp) + s * kTileSlots; };
    const uint32_t k_bytes = Lay::kTile + (p.masked ? 512u : 0u);
    auto load_k = [&](int j) {
        const int s = j % kBStages;
        uint64_t* full = &bars[BB_K_FULL + s];
        mbar_arrive_expect_tx(full, k_bytes);
        bulk_g2s(k_ptr(s), p.kc + (static_cast<size_t>(h) * T + j) * Lay::kTile, Lay::kTile, full);
        if (p.masked) bulk_g2s(grp_ptr(s), p.grp + j * kTileSlots, 512, full);
    };
    auto load_v = [&](int j) {
        const int s = j % kBStages;
        uint64_t* full = &bars[BB_V_FULL + s];
        mbar_arrive_expect_tx(full, Lay::kTile);
        bulk_g2s(v_ptr(s), p.vt + (static_cast<size_t>(h) * T + j) * Lay::kTile, Lay::kTile, full);
    };
    if (warp == kBWarpLoad && lane == 0)
        for (int j = 0; j < kBStages && j < T; ++j) {
            load_k(j);
            load_v(j);
        }

    // ---- query preparation by all eight warps: warp w takes TMEM lane
    // quadrant w % 4 (its rows) and half w / 4 of the dims.  Each thread
    // issues all of its loads at once, rotates its row's pairs at the row's
    // position (fp32), splits them into bf16 hi + lo pieces and packs them two
    // per column into TMEM (the A operand of Q.K; rows past n are zero).
    {
        constexpr int kHalf = D / 2;          // dims per thread
        constexpr int kWords = D / 4;         // packed columns per piece and half
        const int quad = warp & 3, half = warp >> 2;
        const int row = row0 + quad * 32 + lane;
        const uint32_t q_tm = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kBColQ + half * kWords;
        uint4 w[kHalf / 8];
        float4 cs[kHalf / 4];
        if (row < p.n) {
            const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(row) * p.H + h) * D + half * kHalf);
            const float4* crow = reinterpret_cast<const float4*>(p.rope + static_cast<size_t>(row) * (D / 2) + half * kWords);
#pragma unroll
            for (int u = 0; u < kHalf / 8; ++u) w[u] = qrow[u];
#pragma unroll
            for (int u = 0; u < kHalf / 4; ++u) cs[u] = __ldg(crow + u);
        } else {
#pragma unroll
            for (int u = 0; u < kHalf / 8; ++u) w[u] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < kHalf / 4; ++u) cs[u] = make_float4(1.f, 0.f, 1.f, 0.f);
        }
        uint32_t hi[kWords], lo[kWords];
#pragma unroll
        for (int i = 0; i < kWords; ++i) {  // pair i of the half
            const uint32_t bits = reinterpret_cast<const uint32_t*>(w)[i];
            const float4 c4 = cs[i / 2];
            const float c = (i & 1) ? c4.z : c4.x, sn = (i & 1) ? c4.w : c4.y;
            float x, y;
            rotate_pair(__uint_as_float(bits << 16), __uint_as_float(bits & 0xFFFF0000u), c, sn, x, y);
            const __nv_bfloat162 hh = __floats2bfloat162_rn(x, y);
            const __nv_bfloat162 ll = __floats2bfloat162_rn(x - __low2float(hh), y - __high2float(hh));
            hi[i] = *reinterpret_cast<const uint32_t*>(&hh);
            lo[i] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        if constexpr (kWords == 32) {
            tmem_st32(q_tm, hi);
            tmem_st32(q_tm + D / 2, lo);
        } else {
            tmem_st16(q_tm, hi);
            tmem_st16(q_tm + D / 2, lo);
        }
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == kBWarpLoad) {
        // ------------------------------------------------------------ loader
        // One thread serves two queues: a K stage frees when its Q.K finishes,
        // a V buffer only when its P.V does, so it polls both (non-blocking
        // tests) and refills whichever frees first.
        if (lane == 0) {
            int jk = min(kBStages, T), jv = jk;
            uint64_t t0 = global_timer_ns();
            for (uint32_t it = 1; jk < T || jv < T; ++it) {
                bool moved = false;
                if (jk < T && mbar_test(&bars[BB_K_EMPTY + jk % kBStages], ((jk / kBStages) & 1) ^ 1)) {
                    load_k(jk++);
                    moved = true;
                }
                if (jv < T && mbar_test(&bars[BB_V_EMPTY + jv % kBStages], ((jv / kBStages) & 1) ^ 1)) {
                    load_v(jv++);
                    moved = true;
                }
                if (moved) {
                    t0 = global_timer_ns();
                    continue;
                }
                __nanosleep(64);
                if ((it & 15) == 0) {
                    if (*ab.flag) break;
                    if (global_timer_ns() - t0 > ab.limit_ns) {
                        abort_wait(ab, kDevTimeoutLoader);
                        break;
                    }
                }
            }
            if (*ab.flag) {
                // let the copies in flight land before the CTA exits
                for (int q = 0; q < 2; ++q) {
                    const int issued = q == 0 ? jk : jv;
                    uint64_t* full = &bars[q == 0 ? BB_K_FULL : BB_V_FULL];
                    for (int s = 0; s < kBStages && s < issued; ++s) {
                        const int last = ((issued - 1 - s) / kBStages) * kBStages + s;
                        const uint64_t d0 = global_timer_ns();
                        while (!mbar_try_wait(&full[s], (last / kBStages) & 1) && global_timer_ns() - d0 < 100000000ull) {
                        }
                    }
                }
            }
        }
    } else if (warp == kBWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc_qk = instr_desc(kFmtBF16, kFmtBF16, 128, 128);
        const uint32_t idesc_pv = instr_desc(kFmtF16, kFmtF16, 128, D);
        const uint64_t dk0 = smem_desc(smem_u32(k_ptr(0)), 16, 1024, 2);
        const uint64_t dv0 = smem_desc(smem_u32(v_ptr(0)), 16, 1024, 2);
        // S_b = Q_hi K^T + Q_lo K^T, Q from TMEM; K step kk (16 elements):
        // TMEM columns 8 kk of each piece, K tile block kk / 4, bytes 32 (kk % 4)
        auto issue_qk = [&](int j) {
            const uint32_t d_tmem = tmem + kBColS + 128u * (j & 1);
            const uint64_t kb = dk0 + static_cast<uint64_t>(((j % kBStages) * Lay::kTile) >> 4);
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
                    mma_f16_ts(d_tmem, tmem + kBColQ + pc * (D / 2) + kk * 8, kb + (off >> 4), idesc_qk,
                               (pc | kk) != 0);
                }
        };
        auto issue_pv = [&](int j) {
            const uint32_t a_tmem = tmem + kBColS + 128u * (j & 1);
            const uint64_t vb = dv0 + static_cast<uint64_t>(((j % kBStages) * Lay::kTile) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_f16_ts(tmem + kBColO, a_tmem + kk * 8, vb + (((kk >> 2) * (D * 128) + (kk & 3) * 32) >> 4),
                           idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        };
        auto k_ready = [&](int j) -> bool {
            bool r = true;
            if (lane == 0) r = mbar_wait(&bars[BB_K_FULL + j % kBStages], (j / kBStages) & 1, ab, kDevTimeoutMma);
            return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
        };
        const bool leader = lane == 0;
        bool ok = true;
        for (int j = 0; j < 2 && j < T; ++j) {
            ok = ok && k_ready(j);
            if (ok && leader) {
                tc_fence_after();
                issue_qk(j);
                mma_commit(&bars[BB_S_FULL + j]);
                mma_commit(&bars[BB_K_EMPTY + j]);
            }
        }
        // step j: P.V of tile j, then Q.K of tile j + 2 into the same score
        // buffer (queued behind the P.V that reads its P).  The rendezvous
        // also stands for "V tile j and K tile j + 2 landed" (the checker
        // warp's part), so this warp waits on nothing else: an MMA issue
        // blocks while the tensor pipe's queue is full, so every wait here
        // would add to the step.
        for (int j = 0; j < T; ++j) {
            ok = named_barrier_and(kBNbP, kBNbPThreads, ok);
            if (ok && leader) {
                tc_fence_after();
                issue_pv(j);
                mma_commit(&bars[BB_V_EMPTY + j % kBStages]);
                if (j + 2 < T) {
                    issue_qk(j + 2);
                    mma_commit(&bars[BB_S_FULL + (j & 1)]);
                    mma_commit(&bars[BB_K_EMPTY + (j + 2) % kBStages]);
                } else if (j == T - 1) {
                    mma_commit(&bars[BB_O_DONE]);
                }
            }
        }
        if (leader) {
            mma_commit(&bars[BB_DRAIN]);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&bars[BB_DRAIN], 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (warp >= kBWarpSm0 && warp < kBWarpSmEnd) {
        // ------------------------------------------------------------ softmax
        // Each thread owns one row (TMEM lane) of the M tile; scores in log2
        // units x = S * a with a = log2(e)/sqrt(D); P = exp2(x - m) in fp16,
        // with the running max m moved (and O rescaled) only when a tile
        // raises it by more than 8.
        const int quad = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t o_tm = tmem + lane_off + kBColO;
        const float a = p.sm_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const int b = j & 1, s = j % kBStages;
            const uint32_t s_tm = tmem + lane_off + kBColS + 128u * b;
            const int32_t* sgrp = grp_ptr(s);
            const int nvalid = min(kTileSlots, p.C - j * kTileSlots);
            const bool full = ((p.uniform[j >> 6] >> (j & 63)) & 1ull) && nvalid == kTileSlots;
            if (ok && p.masked) ok = warp_wait(&bars[BB_K_FULL + s], (j / kBStages) & 1, ab, kDevTimeoutSoftmax);
            if (ok) ok = warp_wait(&bars[BB_S_FULL + b], (j >> 1) & 1, ab, kDevTimeoutSoftmax);
            if (ok) {
                tc_fence_after();
                if (!full) {
                    // slots past the ring's end, and on a masked ring empty
                    // slots, get a score of -inf in TMEM: exp2 makes their P
                    // exactly 0 and the max ignores them, so every tile takes
                    // the one code path below (a rolled, warp-uniform loop)
#pragma unroll 1
                    for (int c = p.masked ? 0 : nvalid; c < kTileSlots; ++c)
                        if (c >= nvalid || sgrp[c] < 0) tmem_st1(s_tm + c, 0xFF800000u);
                    tmem_st_wait();
                }
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld32_async(s_tm, v0);
                tmem_ld32_async(s_tm + 32, v1);
                tmem_ld32_async(s_tm + 64, v2);
                tmem_ld32_async(s_tm + 96, v3);
                tmem_wait_ld_dep(v0);
                reg_fence(v1);
                reg_fence(v2);
                reg_fence(v3);
                auto cmax = [](const uint32_t (&v)[32]) {
                    float t = -INFINITY;
#pragma unroll
                    for (int k = 0; k < 32; k += 2) t = max3(t, __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
                    return t;
                };
                const float m_tile = fmaxf(fmaxf(cmax(v0), cmax(v1)), fmaxf(cmax(v2), cmax(v3))) * a;
                const bool bump = (m_run == -INFINITY) || (m_tile > m_run + 8.f);
                const float m_new = bump ? fmaxf(m_run, m_tile) : m_run;
                // a row with no valid slot yet keeps m = -inf; its P is 0 and
                // its O and l are 0, so any finite reference point serves
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = (m_run == -INFINITY) ? 0.f : (bump ? ex2(m_run - m_use) : 1.f);
                const float2 a2 = make_float2(a, a), nm2 = make_float2(-m_use, -m_use);
                float2 ls = make_float2(0.f, 0.f);
                auto p_chunk = [&](const uint32_t (&v)[32], uint32_t* pk) {
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const float2 x = fma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), a2, nm2);
                        const float2 q = make_float2(ex2(x.x), ex2(x.y));
                        ls = add2(ls, q);
                        __half2 hh = __floats2half2_rn(q.x, q.y);
                        pk[k / 2] = *reinterpret_cast<uint32_t*>(&hh);
                    }
                };
                uint32_t pa[32], pb[32];
                p_chunk(v0, pa);
                p_chunk(v1, pa + 16);
                tmem_st32(s_tm, pa);
                p_chunk(v2, pb);
                p_chunk(v3, pb + 16);
                tmem_st32(s_tm + 32, pb);
                const float lsum = ls.x + ls.y;
                // an O rescale waits until the previous tile's P.V has landed
                // in O: the release of its V buffer (that phase cannot have
                // been passed, since P.V of tile j + 2 needs this step's P)
                if (__any_sync(0xffffffffu, j > 0 && alpha != 1.f)) {
                    ok = warp_wait(&bars[BB_V_EMPTY + (j - 1) % kBStages], ((j - 1) / kBStages) & 1, ab,
                                   kDevTimeoutSoftmax);
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t v[32];
                            tmem_ld32(o_tm + 32 * c, v);
#pragma unroll
                            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                            tmem_st32(o_tm + 32 * c, v);
                        }
                    }
                }
                tmem_st_wait();
                l_run = l_run * alpha + lsum;
                m_run = m_new;
            }
            __syncwarp();
            if (p.masked && lane == 0) mbar_arrive(&bars[BB_K_EMPTY + s]);
            tc_fence_before();
            __syncwarp();
            ok = named_barrier_and(kBNbP, kBNbPThreads, ok);
        }
        // ---- epilogue: out = O / l
        if (ok) ok = warp_wait(&bars[BB_O_DONE], 0, ab, kDevTimeoutEpilogue);
        if (ok) {
            tc_fence_after();
            const float fin = (l_run > 0.f) ? 1.f / l_run : 0.f;
            // The warp's 32 rows go out through shared memory (the K stages,
            // free once every MMA has finished, which O_DONE marks): each
            // thread parks its row's 32-column chunk, then each store
            // instruction writes 128-byte lines of four rows instead of one
            // 16-byte piece of 32 rows.
            float* stage = reinterpret_cast<float*>(smem + Lay::kK) + (warp - kBWarpSm0) * (32 * 36);
            const int wrow0 = row0 + quad * 32;  // the warp's first query row
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(o_tm + 32 * c, v);
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4*>(stage + lane * 36 + k) =
                        make_float4(__uint_as_float(v[k]) * fin, __uint_as_float(v[k + 1]) * fin,
                                    __uint_as_float(v[k + 2]) * fin, __uint_as_float(v[k + 3]) * fin);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 4 * i + (lane >> 3), q = lane & 7;  // row r of the warp, float4 q
                    const float4 val = *reinterpret_cast<const float4*>(stage + r * 36 + 4 * q);
                    if (wrow0 + r < p.n)
                        *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(wrow0 + r) * p.H + h) * D + 32 * c +
                                                   4 * q) = val;
                }
                __syncwarp();
            }
        }
    } else if (warp == kBWarpCheck) {
        // ------------------------------------------------------------ checker
        // Confirms, for step j, that V tile j and K tile j + 2 have landed,
        // then joins the rendezvous.  Each buffer's previous occupant was
        // confirmed three tiles earlier, so no wait can see a stale phase.
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            bool r = true;
            if (ok && lane == 0) {
                r = mbar_wait(&bars[BB_V_FULL + j % kBStages], (j / kBStages) & 1, ab, kDevTimeoutMma);
                if (r && j + 2 < T)
                    r = mbar_wait(&bars[BB_K_FULL + (j + 2) % kBStages], ((j + 2) / kBStages) & 1, ab, kDevTimeoutMma);
            }
            ok = ok && __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
            ok = named_barrier_and(kBNbP, kBNbPThreads, ok);
        }
    }
    // warp 7 only helps prepare the queries

    // ------------------------------------------------------------ teardown
    // a role's other lanes wait here for its lane 0, so every warp arrives at
    // the CTA barrier converged
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kBWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
static cudaError_t launch_bf16_attention_d(const AttnParams& p, cudaStream_t s) {
    static std::atomic<uint64_t> configured{0};
    constexpr uint32_t smem = BAttnLayout<D>::kAlloc;
    static_assert(smem <= 227 * 1024, "bf16 attention shared memory over the sm_103 limit");
    cudaError_t e = smem_limit_once(bf16_attn_kernel<D>, smem, configured);
    if (e != cudaSuccess) return e;
    dim3 grid((p.n + kBRows - 1) / kBRows, p.H);
    bf16_attn_kernel<D><<<grid, kBAttnThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bf16_attention(const AttnParams& p, int D, cudaStream_t s) {
    return (D == 128) ? launch_bf16_attention_d<128>(p, s) : launch_bf16_attention_d<64>(p, s);
}

}  // namespace rc
