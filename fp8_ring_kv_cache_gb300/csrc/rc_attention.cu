// rc_attention.cu -- K4, the attention call over the FP8 ring (paperdot
// abstract: the 757 new tokens' queries read all 5,788 slots, 240 calls per
// chunk; cpdf.ai "Blackwell, escalabilidade e limites do decodificador": the
// FP8 attention kernel with per-head scales that the B200 build lacked).
//
// One CTA = one head x 256 query rows (two 128-row M tiles), 448 threads:
//   warp 0        loader: one bulk copy per K tile, Vt tile and scale vectors
//                 per 128-slot KV tile, double-buffered (mbarrier + complete_tx)
//   warp 1        MMA issuer (one lane) and TMEM owner (512 columns)
//   warps 2..5    softmax group 0 (rows 0..127; one row per thread / TMEM lane)
//   warps 6..9    softmax group 1 (rows 128..255)
//   warps 10..13  converter: Vt E4M3 tile -> fp16 tile (exact), 128-byte swizzle
// Per KV tile j and M tile i:
//   S_i = Q_i K_j^T on tcgen05 kind::f8f6f4: Q is split into three E4M3 pieces
//         (hi + mid + lo, 12 significant bits) that accumulate into one fp32
//         TMEM tile, so the score error stays inside the tolerance with FP8 K.
//   softmax: score = S * sq_row * sk_slot * log2(e)/sqrt(D); online max and sum
//         in registers; P = exp2(score - max) * sv_slot / max(sv) -> fp16,
//         written back over S in TMEM.
//   O_i += P_i V_j on tcgen05 kind::f16 with P read from TMEM (A operand) and
//         the converted V tile from shared memory (B operand).
// Two M tiles ping-pong so the tensor pipe works on one tile while the other
// is in softmax.  Output: out = O * max(sv) / l, fp32.
#include "rc_device.cuh"
#include "rc_internal.h"

namespace rc {

constexpr int kAttnWarps = 14;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kQPieces = 3;
constexpr int kStages = 2;
constexpr int kMTile = 128;
constexpr int kRowsPerCta = 2 * kMTile;
constexpr int kWarpLoad = 0, kWarpMma = 1, kWarpSm0 = 2, kWarpCvt = 10;
constexpr uint32_t kTmemCols = 512;

// barrier indices
enum : int {
    B_KV_FULL = 0,   // [2]
    B_KV_EMPTY = 2,  // [2]
    B_V16_FULL = 4,
    B_V16_EMPTY = 5,
    B_S_FULL = 6,    // [2]
    B_P_FULL = 8,    // [2]
    B_O_DONE = 10,   // [2]
    B_DRAIN = 12,
    B_COUNT = 13
};

template <int D>
struct AttnLayout {
    static constexpr uint32_t kTile = kTileSlots * D;  // bytes of a K tile or a Vt tile
    static constexpr uint32_t kQ = 0;                   // [piece][mtile][128][D] E4M3
    static constexpr uint32_t kQBytes = kQPieces * 2 * kMTile * D;
    static constexpr uint32_t kStage0 = kQBytes;        // K8, V8, sk[128], sv[128], grp[128]
    static constexpr uint32_t kStageBytes = ((2 * kTile + 3 * 512) + 1023) / 1024 * 1024;
    static constexpr uint32_t kV16 = kStage0 + kStages * kStageBytes;  // [2 halves][D][128 B] fp16
    static constexpr uint32_t kV16Bytes = 2 * D * 128;
    static constexpr uint32_t kBar = kV16 + kV16Bytes;
    static constexpr uint32_t kMisc = kBar + 8 * 16;
    static constexpr uint32_t kTotal = kMisc + 64;
    static constexpr uint32_t kAlloc = kTotal + 1024;  // room to align the base to 1024
};

// Every lane waits; the warp continues only if all lanes saw the phase.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, AbortState ab, int where) {
    const bool ok = mbar_wait(bar, parity, ab, where);
    return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(AttnParams p) {
    using Lay = AttnLayout<D>;
    constexpr uint32_t kSboK = (D == 128) ? 1024u : 512u;  // 8 rows of D bytes
    constexpr uint32_t kSwzK = (D == 128) ? 2u : 4u;       // 128-byte / 64-byte swizzle
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);  // [0] tmem, [1] svmax, [2] abort

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int row0 = blockIdx.x * kRowsPerCta;
    const int T = p.T;
    AbortState ab{reinterpret_cast<volatile uint32_t*>(&misc[2]), p.status};

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[B_KV_FULL + s], 1);
            mbar_init(&bars[B_KV_EMPTY + s], 1 + 4 + 8);
        }
        mbar_init(&bars[B_V16_FULL], 4);
        mbar_init(&bars[B_V16_EMPTY], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_S_FULL + i], 1);
            mbar_init(&bars[B_P_FULL + i], 4);
            mbar_init(&bars[B_O_DONE + i], 1);
        }
        mbar_init(&bars[B_DRAIN], 1);
        misc[1] = 0u;
        misc[2] = 0u;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&misc[0], kTmemCols);
        tmem_relinquish();
    }

    // softmax groups: rotate their Q rows, split into three E4M3 pieces
    const bool is_sm = (warp >= kWarpSm0) && (warp < kWarpSm0 + 8);
    const int mt = is_sm ? (warp - kWarpSm0) >> 2 : 0;    // M tile of this softmax group
    const int quad = warp & 3;                             // TMEM lane quadrant
    const int r = quad * 32 + lane;                        // row within the M tile
    const int grow = row0 + mt * kMTile + r;               // query row
    float qscale = 1.f;
    if (is_sm) {
        uint8_t* qdst[kQPieces];
#pragma unroll
        for (int pc = 0; pc < kQPieces; ++pc) qdst[pc] = smem + Lay::kQ + (pc * 2 + mt) * (kMTile * D);
        if (grow < p.n) {
            const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(grow) * p.H + h) * D;
            const float2* rrow = p.rope + static_cast<size_t>(grow) * (D / 2);
            float amax = 0.f;
            for (int c = 0; c < D / 16; ++c) {
                uint4 qa = *reinterpret_cast<const uint4*>(qrow + c * 16);
                uint4 qb = *reinterpret_cast<const uint4*>(qrow + c * 16 + 8);
                const __nv_bfloat16* qv0 = reinterpret_cast<const __nv_bfloat16*>(&qa);
                const __nv_bfloat16* qv1 = reinterpret_cast<const __nv_bfloat16*>(&qb);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 cs = rrow[c * 8 + j];
                    const __nv_bfloat16* src = (j < 4) ? qv0 : qv1;
                    float x, y;
                    rotate_pair(__bfloat162float(src[(2 * j) & 7]), __bfloat162float(src[(2 * j + 1) & 7]), cs.x,
                                cs.y, x, y);
                    amax = fmaxf(amax, fmaxf(fabsf(x), fabsf(y)));
                }
            }
            qscale = (amax > 0.f) ? __fdiv_rn(amax, 448.f) : 1.f;
            const float inv = __frcp_rn(qscale);
            for (int c = 0; c < D / 16; ++c) {
                uint4 qa = *reinterpret_cast<const uint4*>(qrow + c * 16);
                uint4 qb = *reinterpret_cast<const uint4*>(qrow + c * 16 + 8);
                const __nv_bfloat16* qv0 = reinterpret_cast<const __nv_bfloat16*>(&qa);
                const __nv_bfloat16* qv1 = reinterpret_cast<const __nv_bfloat16*>(&qb);
                uint32_t w[kQPieces][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 cs = rrow[c * 8 + j];
                    const __nv_bfloat16* src = (j < 4) ? qv0 : qv1;
                    float x, y;
                    rotate_pair(__bfloat162float(src[(2 * j) & 7]), __bfloat162float(src[(2 * j + 1) & 7]), cs.x,
                                cs.y, x, y);
                    float rx = x * inv, ry = y * inv;
#pragma unroll
                    for (int pc = 0; pc < kQPieces; ++pc) {
                        const uint32_t two = e4m3x2(rx, ry);
                        const float2 back = e4m3x2_to_float2(static_cast<uint16_t>(two));
                        rx -= back.x;
                        ry -= back.y;
                        if ((j & 1) == 0)
                            w[pc][j >> 1] = two;
                        else
                            w[pc][j >> 1] |= two << 16;
                    }
                }
#pragma unroll
                for (int pc = 0; pc < kQPieces; ++pc)
                    *reinterpret_cast<uint4*>(qdst[pc] + ktile_off(r, c * 16, D)) =
                        make_uint4(w[pc][0], w[pc][1], w[pc][2], w[pc][3]);
            }
        } else {
            for (int c = 0; c < D / 16; ++c)
#pragma unroll
                for (int pc = 0; pc < kQPieces; ++pc)
                    *reinterpret_cast<uint4*>(qdst[pc] + ktile_off(r, c * 16, D)) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();  // the MMA reads these rows through the async proxy
    }
    // converter group: the head's largest V scale (the P.V operand reference)
    if (warp >= kWarpCvt) {
        float m = 0.f;
        for (int i = tid - kWarpCvt * 32; i < p.C; i += 128) m = fmaxf(m, p.sv[static_cast<size_t>(h) * p.Cpad + i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) atomicMax(&misc[1], __float_as_uint(m));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const float svmax = __uint_as_float(misc[1]);

    auto stage_ptr = [&](int s) { return smem + Lay::kStage0 + s * Lay::kStageBytes; };

    if (warp == kWarpLoad) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            const uint32_t bytes = 2 * Lay::kTile + 1024 + (p.masked ? 512 : 0);
            for (int j = 0; j < T; ++j) {
                const int s = j & 1;
                if (!mbar_wait(&bars[B_KV_EMPTY + s], ((j >> 1) & 1) ^ 1, ab, kDevTimeoutLoader)) break;
                uint8_t* st = stage_ptr(s);
                uint64_t* full = &bars[B_KV_FULL + s];
                mbar_arrive_expect_tx(full, bytes);
                bulk_g2s(st, p.kc + (static_cast<size_t>(h) * T + j) * Lay::kTile, Lay::kTile, full);
                bulk_g2s(st + Lay::kTile, p.vt + (static_cast<size_t>(h) * T + j) * Lay::kTile, Lay::kTile, full);
                bulk_g2s(st + 2 * Lay::kTile, p.sk + static_cast<size_t>(h) * p.Cpad + j * kTileSlots, 512, full);
                bulk_g2s(st + 2 * Lay::kTile + 512, p.sv + static_cast<size_t>(h) * p.Cpad + j * kTileSlots, 512,
                         full);
                if (p.masked) bulk_g2s(st + 2 * Lay::kTile + 1024, p.grp + j * kTileSlots, 512, full);
            }
            if (*ab.flag) {
                // leave no copy in flight: wait (bounded) for the last fill of each stage
                AbortState quiet{ab.flag, ab.status};
                for (int s = 0; s < kStages && s < T; ++s) {
                    const int last = ((T - 1 - s) / kStages) * kStages + s;
                    uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(&bars[B_KV_FULL + s], (last >> 1) & 1) &&
                           global_timer_ns() - t0 < 100000000ull) {
                    }
                    (void)quiet;
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = instr_desc(kFmtE4M3, kFmtE4M3, 128, 128);
            const uint32_t idesc_pv = instr_desc(kFmtF16, kFmtF16, 128, D);
            const uint32_t q_base = smem_u32(smem + Lay::kQ);
            const uint32_t v16_base = smem_u32(smem + Lay::kV16);
            auto issue_qk = [&](int i, int s) {
                const uint32_t k_base = smem_u32(stage_ptr(s));
                const uint32_t d_tmem = tmem + 128u * i;
#pragma unroll
                for (int pc = 0; pc < kQPieces; ++pc)
#pragma unroll
                    for (int k = 0; k < D / 32; ++k) {
                        const uint64_t a = smem_desc(q_base + (pc * 2 + i) * (kMTile * D) + k * 32, 16, kSboK, kSwzK);
                        const uint64_t b = smem_desc(k_base + k * 32, 16, kSboK, kSwzK);
                        mma_f8_ss(d_tmem, a, b, idesc_qk, (pc | k) != 0);
                    }
            };
            auto issue_pv = [&](int i, bool acc) {
                const uint32_t d_tmem = tmem + 256u + static_cast<uint32_t>(D) * i;
                const uint32_t a_tmem = tmem + 128u * i;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t b = smem_desc(v16_base + (kk >> 2) * (D * 128) + (kk & 3) * 32, 16, 1024, 2);
                    mma_f16_ts(d_tmem, a_tmem + kk * 8, b, idesc_pv, (acc || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            for (int j = 0; j < T && ok; ++j) {
                const int s = j & 1;
                ok = mbar_wait(&bars[B_KV_FULL + s], (j >> 1) & 1, ab, kDevTimeoutMma);
                if (!ok) break;
                tc_fence_after();
                for (int i = 0; i < 2 && ok; ++i) {
                    if (j > 0) {
                        ok = mbar_wait(&bars[B_P_FULL + i], (j - 1) & 1, ab, kDevTimeoutMma);
                        if (ok && i == 0) ok = mbar_wait(&bars[B_V16_FULL], (j - 1) & 1, ab, kDevTimeoutMma);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(i, j - 1 > 0);
                        if (i == 1) mma_commit(&bars[B_V16_EMPTY]);
                    }
                    issue_qk(i, s);
                    mma_commit(&bars[B_S_FULL + i]);
                }
                if (ok) mma_commit(&bars[B_KV_EMPTY + s]);
            }
            for (int i = 0; i < 2 && ok; ++i) {
                ok = mbar_wait(&bars[B_P_FULL + i], (T - 1) & 1, ab, kDevTimeoutMma);
                if (ok && i == 0) ok = mbar_wait(&bars[B_V16_FULL], (T - 1) & 1, ab, kDevTimeoutMma);
                if (!ok) break;
                tc_fence_after();
                issue_pv(i, T - 1 > 0);
                mma_commit(&bars[B_O_DONE + i]);
            }
            // every MMA has finished before the tensor memory is released
            mma_commit(&bars[B_DRAIN]);
            uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&bars[B_DRAIN], 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (is_sm) {
        // ------------------------------------------------------------ softmax
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t s_tm = tmem + lane_off + 128u * mt;
        const uint32_t o_tm = tmem + lane_off + 256u + static_cast<uint32_t>(D) * mt;
        const float a = qscale * p.sm_log2;  // > 0
        const float inv_svmax = (svmax > 0.f) ? __frcp_rn(svmax) : 1.f;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const int s = j & 1;
            ok = warp_wait(&bars[B_S_FULL + mt], j & 1, ab, kDevTimeoutSoftmax);
            if (ok) ok = warp_wait(&bars[B_KV_FULL + s], (j >> 1) & 1, ab, kDevTimeoutSoftmax);
            if (!ok) break;
            tc_fence_after();
            const uint8_t* st = stage_ptr(s);
            const float* ssk = reinterpret_cast<const float*>(st + 2 * Lay::kTile);
            const float* ssv = ssk + kTileSlots;
            const int32_t* sgrp = reinterpret_cast<const int32_t*>(ssv + kTileSlots);
            const int nvalid = min(kTileSlots, p.C - j * kTileSlots);
            const bool full = (nvalid == kTileSlots) && !p.masked;
            auto valid = [&](int col) { return full || (col < nvalid && (!p.masked || sgrp[col] >= 0)); };
            // pass A: the tile's largest scaled score
            float mx = -INFINITY;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld32(s_tm + 32 * c, v);
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int col = 32 * c + k;
                    const float x = valid(col) ? __uint_as_float(v[k]) * ssk[col] : -INFINITY;
                    mx = fmaxf(mx, x);
                }
            }
            const float m_new = fmaxf(m_run, mx * a);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m_run - m_use);
            // pass B: probabilities, row sum, fp16 P (with the V scale) over S
            float l_tile = 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld32(s_tm + 32 * c, v);
                uint32_t pk[16];
#pragma unroll
                for (int k2 = 0; k2 < 16; ++k2) {
                    const int c0 = 32 * c + 2 * k2, c1 = c0 + 1;
                    const float p0 = valid(c0) ? ex2(__fmaf_rn(__uint_as_float(v[2 * k2]) * ssk[c0], a, -m_use)) : 0.f;
                    const float p1 = valid(c1) ? ex2(__fmaf_rn(__uint_as_float(v[2 * k2 + 1]) * ssk[c1], a, -m_use)) : 0.f;
                    l_tile += p0 + p1;
                    __half2 hp = __floats2half2_rn(p0 * (ssv[c0] * inv_svmax), p1 * (ssv[c1] * inv_svmax));
                    pk[k2] = *reinterpret_cast<uint32_t*>(&hp);
                }
                tmem_st16(s_tm + 16 * c, pk);
            }
            tmem_st_wait();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_KV_EMPTY + s]);
            // rescale the running output when the max moved (warp-uniform)
            if (__any_sync(0xffffffffu, j > 0 && alpha != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_tm + 32 * c, v);
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                    tmem_st32(o_tm + 32 * c, v);
                }
                tmem_st_wait();
            }
            l_run = l_run * alpha + l_tile;
            m_run = m_new;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_P_FULL + mt]);
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = warp_wait(&bars[B_O_DONE + mt], 0, ab, kDevTimeoutEpilogue);
        if (ok) {
            tc_fence_after();
            const float fin = (l_run > 0.f) ? svmax / l_run : 0.f;
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
    } else if (warp >= kWarpCvt) {
        // ------------------------------------------------------------ V converter
        const int ct = tid - kWarpCvt * 32;
        uint8_t* v16 = smem + Lay::kV16;
        for (int j = 0; j < T; ++j) {
            const int s = j & 1;
            bool ok = warp_wait(&bars[B_KV_FULL + s], (j >> 1) & 1, ab, kDevTimeoutConvert);
            if (ok) ok = warp_wait(&bars[B_V16_EMPTY], (j & 1) ^ 1, ab, kDevTimeoutConvert);
            if (!ok) break;
            const uint8_t* v8 = stage_ptr(s) + Lay::kTile;
#pragma unroll 2
            for (int u = ct; u < D * 8; u += 128) {
                const int rr = u >> 3, cp = u & 7;
                const uint4 raw = *reinterpret_cast<const uint4*>(v8 + rr * 128 + cp * 16);
                const int c = cp ^ (rr & 7);  // logical 16-slot chunk
                const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t o[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    __half2_raw lo = e4m3x2_to_half2(static_cast<uint16_t>(in[q] & 0xFFFFu));
                    __half2_raw hi = e4m3x2_to_half2(static_cast<uint16_t>(in[q] >> 16));
                    o[2 * q] = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
                    o[2 * q + 1] = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
                }
                uint8_t* dst = v16 + (c >> 2) * (D * 128) + rr * 128;
                const int l0 = 2 * (c & 3);
                *reinterpret_cast<uint4*>(dst + (((l0) ^ (rr & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(dst + (((l0 + 1) ^ (rr & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_V16_FULL]);
                mbar_arrive(&bars[B_KV_EMPTY + s]);
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
static cudaError_t launch_attention_d(const AttnParams& p, cudaStream_t s) {
    static bool configured = false;
    constexpr uint32_t smem = AttnLayout<D>::kAlloc;
    static_assert(smem <= 227 * 1024, "attention shared memory over the sm_103 limit");
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid((p.n + kRowsPerCta - 1) / kRowsPerCta, p.H);
    attn_kernel<D><<<grid, kAttnThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_attention(const AttnParams& p, int D, cudaStream_t s) {
    return (D == 128) ? launch_attention_d<128>(p, s) : launch_attention_d<64>(p, s);
}

}  // namespace rc
