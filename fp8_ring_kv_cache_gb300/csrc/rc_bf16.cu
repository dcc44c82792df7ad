// rc_bf16.cu -- the same path with a bf16 ring (RC_F_BF16_CACHE): the non-FP8
// cache of the comparison the cpdf.ai blog draws in "Blackwell, escalabilidade
// e limites do decodificador" (the FP8 cache saved 17.0 ms a step on H100 and
// cost 2.4-6.7 ms on B200, whose build had no per-head-scaled FP8 attention).
// Keys are still rotated once, at write time, and re-rotated on a position
// reset; only the storage differs: one bf16 rounding instead of per-head E4M3.
//
// KB1 bf16_write_kernel: K rotated by RoPE (fp32, fp64-angle cos/sin) and
//    rounded once to bf16 into the K tile; V copied bit for bit into the
//    transposed Vt tile through a shared-memory transpose.
// KB2 bf16_rotate_kernel: every stored key of every layer re-rotated by the
//    delta and rounded to bf16 again, in place (no scales to recompute).
// KB3 bf16_attn_kernel: one CTA = one head x 128 query rows.  The queries are
//    rotated and split into two bf16 pieces (hi + lo, ~16 significant bits);
//    S = Q K^T on tcgen05 kind::f16 (bf16 operands, two MMAs per K step), P in
//    fp16, O += P V on kind::f16 with V converted exactly to fp16 in shared
//    memory.  The scores are double-buffered in TMEM over KV tiles: Q.K of
//    tile j + 2 is queued behind P.V of tile j, so the tensor pipe works while
//    the softmax processes the next tile.  Warps: 0 loader (K tiles by bulk
//    copy), 1 MMA issuer, 2..5 softmax (one TMEM lane quadrant each), 6..7 V
//    converters.
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
    __shared__ __align__(16) __nv_bfloat16 vs[kBWriteTokens][D + 8];
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
        for (int e = 0; e < EPL; ++e) vs[tl][dim0 + e] = vb[e];
        if (lane == 0 && h == 0) p.grp[slot] = p.group;
    }
    __syncthreads();
    // V transposed: a warp per dim row, the lanes over the tokens, so each store
    // instruction writes the consecutive slots of one dim row
    uint8_t* vhead = p.vt + static_cast<size_t>(h) * p.T * (kTileSlots * D * 2);
    for (int d = warp; d < D; d += kBWriteThreads / 32) {
        for (int tl = lane; tl < cnt; tl += 32) {
            const int slot = s_slot[tl];
            *reinterpret_cast<__nv_bfloat16*>(vhead + static_cast<size_t>(slot >> 7) * (kTileSlots * D * 2) +
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
constexpr int kBWarpLoad = 0, kBWarpMma = 1, kBWarpSm0 = 2, kBWarpCvt = 6, kBCvtWarps = 2;
constexpr int kBNbP = 1;                           // named barrier: P of a tile is in TMEM
constexpr int kBNbPThreads = 4 * 32 + 32;

enum : int {
    BB_KV_FULL = 0,    // [2] K tile (and the tile's write groups) landed
    BB_KV_EMPTY = 2,   // [2] its Q.K finished and the 4 softmax warps read the groups
    BB_V16_FULL = 4,   // [2] fp16 V buffer filled
    BB_V16_EMPTY = 6,  // [2] its P.V finished
    BB_S_FULL = 8,     // [2] scores of a tile in TMEM score buffer b
    BB_O_READY = 10,   // one completion per P.V (the softmax waits on it before an O rescale)
    BB_O_DONE = 11,
    BB_DRAIN = 12,
    BB_COUNT = 13
};

template <int D>
struct BAttnLayout {
    static constexpr uint32_t kTile = kTileSlots * D * 2;   // bytes of a bf16 K or Vt tile
    static constexpr uint32_t kQ = 0;                        // [2 pieces][D/64][128][128 B] bf16
    static constexpr uint32_t kQBytes = 2 * kBRows * D * 2;
    static constexpr uint32_t kStage0 = kQBytes;             // K tile | grp[128]
    static constexpr uint32_t kStageBytes = ((kTile + 512) + 1023) / 1024 * 1024;
    static constexpr uint32_t kV16 = kStage0 + 2 * kStageBytes;  // 2 x [2 halves][D][128 B] fp16
    static constexpr uint32_t kV16One = kTile;
    static constexpr uint32_t kBar = kV16 + 2 * kV16One;
    static constexpr uint32_t kMisc = kBar + 8 * BB_COUNT;
    static constexpr uint32_t kTotal = kMisc + 64;
    static constexpr uint32_t kAlloc = kTotal + 1024;
};

// Softmax of a tile that is not entirely occupied (a partially filled ring or
// the ring's last tile): the scores of empty or missing slots are cut, the row
// max and P computed per 32-column chunk.  Returns (tile max in log2 units,
// row sum of P); P (fp16) goes to TMEM columns 0..63.  Kept out of line.
__device__ __noinline__ float2 bf16_masked_tile(uint32_t s_tm, const int32_t* sgrp, int masked, int nvalid, float a,
                                                float m_fixed, bool max_only) {
    float mx = -INFINITY, sum = 0.f;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(s_tm + 32 * c, v);
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
            const int col = 32 * c + k;
            const bool ok0 = col < nvalid && (!masked || sgrp[col] >= 0);
            const bool ok1 = col + 1 < nvalid && (!masked || sgrp[col + 1] >= 0);
            const float x0 = __uint_as_float(v[k]) * a, x1 = __uint_as_float(v[k + 1]) * a;
            if (max_only) {
                mx = max3(mx, ok0 ? x0 : -INFINITY, ok1 ? x1 : -INFINITY);
            } else {
                const float q0 = ok0 ? ex2(x0 - m_fixed) : 0.f, q1 = ok1 ? ex2(x1 - m_fixed) : 0.f;
                sum += q0 + q1;
                __half2 hh = __floats2half2_rn(q0, q1);
                pk[k / 2] = *reinterpret_cast<uint32_t*>(&hh);
            }
        }
        if (!max_only) tmem_st16(s_tm + 16 * c, pk);
    }
    return make_float2(mx, sum);
}

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
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[BB_KV_FULL + b], 1);
            mbar_init(&bars[BB_KV_EMPTY + b], 1 + 4);
            mbar_init(&bars[BB_V16_FULL + b], kBCvtWarps);
            mbar_init(&bars[BB_V16_EMPTY + b], 1);
            mbar_init(&bars[BB_S_FULL + b], 1);
        }
        mbar_init(&bars[BB_O_READY], 1);
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
    const uint32_t tmem = misc[0];  // S buffers at columns 0 and 128, O at 256

    auto stage_ptr = [&](int s) { return smem + Lay::kStage0 + s * Lay::kStageBytes; };
    const uint32_t kv_bytes = Lay::kTile + (p.masked ? 512u : 0u);
    auto load_tile = [&](int j) {
        const int s = j & 1;
        uint64_t* full = &bars[BB_KV_FULL + s];
        mbar_arrive_expect_tx(full, kv_bytes);
        bulk_g2s(stage_ptr(s), p.kc + (static_cast<size_t>(h) * T + j) * Lay::kTile, Lay::kTile, full);
        if (p.masked) bulk_g2s(stage_ptr(s) + Lay::kTile, p.grp + j * kTileSlots, 512, full);
    };
    if (warp == kBWarpLoad && lane == 0)
        for (int j = 0; j < 2 && j < T; ++j) load_tile(j);

    // ---- query preparation: rows staged in the V buffers, rotated at their
    // positions (fp32) and split into bf16 hi + lo pieces in the A-operand image
    {
        uint8_t* qstage = smem + Lay::kV16;  // [128 rows][D] bf16, 16-byte pieces XOR-swizzled by row
        constexpr int kUnits = D * 2 / 16;
        const int rows_here = min(kBRows, p.n - row0);
        for (int u = tid; u < rows_here * kUnits; u += kBAttnThreads) {
            const int rr = u / kUnits, c = u - rr * kUnits;
            cp_async16(qstage + rr * (D * 2) + ((c ^ (rr & 7)) << 4),
                       p.q + (static_cast<size_t>(row0 + rr) * p.H + h) * D + c * 8);
        }
        cp_async_wait_all();
        __syncthreads();
        // a thread per (row, 8-dim chunk)
        for (int u = tid; u < kBRows * (D / 8); u += kBAttnThreads) {
            const int rr = u / (D / 8), c = u - rr * (D / 8);
            const int row = row0 + rr;
            float x[8];
            if (row < p.n) {
                const uint4 w = *reinterpret_cast<const uint4*>(qstage + rr * (D * 2) + ((c ^ (rr & 7)) << 4));
                const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(&w);
                const float2* cs = p.rope + static_cast<size_t>(row) * (D / 2) + c * 4;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 r2 = __ldg(cs + j);
                    rotate_pair(__bfloat162float(qb[2 * j]), __bfloat162float(qb[2 * j + 1]), r2.x, r2.y, x[2 * j],
                                x[2 * j + 1]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = 0.f;
            }
            __nv_bfloat16 hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                hi[e] = __float2bfloat16_rn(x[e]);
                lo[e] = __float2bfloat16_rn(x[e] - __bfloat162float(hi[e]));
            }
            const uint32_t off = bktile_off(rr, c * 8);
            *reinterpret_cast<uint4*>(smem + Lay::kQ + off) = *reinterpret_cast<const uint4*>(hi);
            *reinterpret_cast<uint4*>(smem + Lay::kQ + kBRows * D * 2 + off) = *reinterpret_cast<const uint4*>(lo);
        }
        fence_async_smem();
    }
    __syncthreads();

    if (warp == kBWarpLoad) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            for (int j = 2; j < T; ++j) {
                const int s = j & 1;
                if (!mbar_wait(&bars[BB_KV_EMPTY + s], ((j >> 1) & 1) ^ 1, ab, kDevTimeoutLoader)) break;
                load_tile(j);
            }
            if (*ab.flag) {
                for (int s = 0; s < 2 && s < T; ++s) {
                    const int last = ((T - 1 - s) / 2) * 2 + s;
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(&bars[BB_KV_FULL + s], (last >> 1) & 1) &&
                           global_timer_ns() - t0 < 100000000ull) {
                    }
                }
            }
        }
    } else if (warp == kBWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc_qk = instr_desc(kFmtBF16, kFmtBF16, 128, 128);
        const uint32_t idesc_pv = instr_desc(kFmtF16, kFmtF16, 128, D);
        const uint64_t dq0 = smem_desc(smem_u32(smem + Lay::kQ), 16, 1024, 2);
        const uint64_t dk0 = smem_desc(smem_u32(stage_ptr(0)), 16, 1024, 2);
        const uint64_t dv0 = smem_desc(smem_u32(smem + Lay::kV16), 16, 1024, 2);
        // S_b = Q_hi K^T + Q_lo K^T; K step kk (16 elements): block kk / 4, bytes 32 (kk % 4)
        auto issue_qk = [&](int j) {
            const uint32_t d_tmem = tmem + 128u * (j & 1);
            const uint64_t kb = dk0 + static_cast<uint64_t>(((j & 1) * Lay::kStageBytes) >> 4);
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
                    mma_f16_ss(d_tmem, dq0 + ((pc * kBRows * D * 2 + off) >> 4), kb + (off >> 4), idesc_qk,
                               (pc | kk) != 0);
                }
        };
        auto issue_pv = [&](int j) {
            const uint32_t a_tmem = tmem + 128u * (j & 1);
            const uint64_t vb = dv0 + static_cast<uint64_t>(((j & 1) * Lay::kV16One) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_f16_ts(tmem + 256u, a_tmem + kk * 8, vb + (((kk >> 2) * (D * 128) + (kk & 3) * 32) >> 4),
                           idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        };
        auto kv_ready = [&](int j) -> bool {
            bool r = true;
            if (lane == 0) r = mbar_wait(&bars[BB_KV_FULL + (j & 1)], (j >> 1) & 1, ab, kDevTimeoutMma);
            return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
        };
        const bool leader = lane == 0;
        bool ok = true;
        for (int j = 0; j < 2 && j < T; ++j) {
            ok = ok && kv_ready(j);
            if (ok && leader) {
                tc_fence_after();
                issue_qk(j);
                mma_commit(&bars[BB_S_FULL + j]);
                mma_commit(&bars[BB_KV_EMPTY + j]);
            }
        }
        // step j: P.V of tile j, then Q.K of tile j + 2 into the same score
        // buffer (queued behind the P.V that reads its P).  The P rendezvous
        // also stands for "fp16 V of tile j converted" and "K tile j + 2 landed"
        // (tested by a softmax lane), so this warp polls nothing in the loop.
        for (int j = 0; j < T; ++j) {
            ok = named_barrier_and(kBNbP, kBNbPThreads, ok);
            if (ok && leader) {
                tc_fence_after();
                issue_pv(j);
                mma_commit(&bars[BB_V16_EMPTY + (j & 1)]);
                mma_commit(&bars[BB_O_READY]);
                if (j + 2 < T) {
                    issue_qk(j + 2);
                    mma_commit(&bars[BB_S_FULL + (j & 1)]);
                    mma_commit(&bars[BB_KV_EMPTY + (j & 1)]);
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
    } else if (warp < kBWarpCvt) {
        // ------------------------------------------------------------ softmax
        // Row r (TMEM lane) of the M tile; scores in log2 units x = S * a with
        // a = log2(e)/sqrt(D); P = exp2(x - m) in fp16, with the running max m
        // moved (and O rescaled) only when a tile raises it by more than 8.
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int grow = row0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t o_tm = tmem + lane_off + 256u;
        const float a = p.sm_log2;
        const bool checker = warp == kBWarpSm0 && lane == 0;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const int b = j & 1;
            const uint32_t s_tm = tmem + lane_off + 128u * b;
            const int32_t* sgrp = reinterpret_cast<const int32_t*>(stage_ptr(b) + Lay::kTile);
            const int nvalid = min(kTileSlots, p.C - j * kTileSlots);
            const bool full = ((p.uniform[j >> 6] >> (j & 63)) & 1ull) && nvalid == kTileSlots;
            if (ok) ok = warp_wait(&bars[BB_KV_FULL + b], (j >> 1) & 1, ab, kDevTimeoutSoftmax);
            // the checker lane tests fp16 V of tile j and K tile j + 2 now and
            // reads the answers after the softmax.  The K test must follow the
            // wait on tile j, which shares the stage: before tile j's phase
            // completes, a test of the next phase's parity reports the phase
            // before it and would pass early.
            bool vk = true;
            if (checker && ok) {
                vk = mbar_test(&bars[BB_V16_FULL + b], (j >> 1) & 1);
                if (j + 2 < T) vk = mbar_test(&bars[BB_KV_FULL + b], ((j + 2) >> 1) & 1) && vk;
            }
            if (ok) ok = warp_wait(&bars[BB_S_FULL + b], (j >> 1) & 1, ab, kDevTimeoutSoftmax);
            if (ok) {
                tc_fence_after();
                float m_new = m_run, alpha = 1.f, lsum = 0.f;
                if (full) {
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
                    m_new = bump ? fmaxf(m_run, m_tile) : m_run;
                    alpha = bump ? ex2(m_run - m_new) : 1.f;
                    const float2 a2 = make_float2(a, a), nm2 = make_float2(-m_new, -m_new);
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
                    lsum = ls.x + ls.y;
                } else {
                    const float2 mt = bf16_masked_tile(s_tm, sgrp, p.masked, nvalid, a, 0.f, true);
                    const bool bump = (m_run == -INFINITY) || (mt.x > m_run + 8.f);
                    m_new = bump ? fmaxf(m_run, mt.x) : m_run;
                    const float m_fin = (m_new == -INFINITY) ? 0.f : m_new;
                    alpha = bump ? ex2(m_run - m_fin) : 1.f;
                    lsum = bf16_masked_tile(s_tm, sgrp, p.masked, nvalid, a, m_fin, false).y;
                }
                // an O rescale waits until the previous tile's P.V has landed in O
                if (__any_sync(0xffffffffu, j > 0 && alpha != 1.f)) {
                    ok = warp_wait(&bars[BB_O_READY], (j - 1) & 1, ab, kDevTimeoutSoftmax);
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
            if (lane == 0) mbar_arrive(&bars[BB_KV_EMPTY + b]);
            if (checker && ok && !vk) {
                ok = mbar_wait(&bars[BB_V16_FULL + b], (j >> 1) & 1, ab, kDevTimeoutSoftmax);
                if (ok && j + 2 < T) ok = mbar_wait(&bars[BB_KV_FULL + b], ((j + 2) >> 1) & 1, ab, kDevTimeoutSoftmax);
            }
            tc_fence_before();
            __syncwarp();
            ok = named_barrier_and(kBNbP, kBNbPThreads, ok);
        }
        // ---- epilogue: out = O / l
        if (ok) ok = warp_wait(&bars[BB_O_DONE], 0, ab, kDevTimeoutEpilogue);
        if (ok) {
            tc_fence_after();
            const float fin = (l_run > 0.f) ? 1.f / l_run : 0.f;
            float* orow = p.out + (static_cast<size_t>(grow) * p.H + h) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(o_tm + 32 * c, v);
                if (grow < p.n) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4*>(orow + 32 * c + k) =
                            make_float4(__uint_as_float(v[k]) * fin, __uint_as_float(v[k + 1]) * fin,
                                        __uint_as_float(v[k + 2]) * fin, __uint_as_float(v[k + 3]) * fin);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ V converter
        // The bf16 Vt tile and the fp16 buffer share one layout: each 16-byte
        // piece is converted in place of its copy (exact for |v| < 65504).
        constexpr int kCvtThreads = kBCvtWarps * 32;
        const int ct = tid - kBWarpCvt * 32;
        const uint8_t* vhead = p.vt + static_cast<size_t>(h) * T * Lay::kTile;
        bool cok = true;
        for (int j = 0; j < T; ++j) {
            const int b = j & 1;
            if (j >= 2 && cok) cok = warp_wait(&bars[BB_V16_EMPTY + b], ((j >> 1) & 1) ^ 1, ab, kDevTimeoutConvert);
            if (!cok) break;
            const uint8_t* src = vhead + static_cast<size_t>(j) * Lay::kTile;
            uint8_t* dst = smem + Lay::kV16 + b * Lay::kV16One;
#pragma unroll 4
            for (int u = ct; u < static_cast<int>(Lay::kTile / 16); u += kCvtThreads) {
                const uint4 w = ldg_nc_na_v4(src + u * 16);
                const uint32_t in[4] = {w.x, w.y, w.z, w.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float lo = __uint_as_float(in[q] << 16), hi = __uint_as_float(in[q] & 0xFFFF0000u);
                    __half2 hh = __floats2half2_rn(lo, hi);
                    o[q] = *reinterpret_cast<uint32_t*>(&hh);
                }
                *reinterpret_cast<uint4*>(dst + u * 16) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BB_V16_FULL + b]);
        }
    }

    // ------------------------------------------------------------ teardown
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
