// rc_attention.cu -- the attention call over the FP8 ring (paperdot abstract:
// the 757 new tokens' queries read all 5,788 slots, 240 calls per chunk;
// cpdf.ai "Blackwell, escalabilidade e limites do decodificador": the FP8
// attention kernel with per-head scales that the B200 build lacked).
//
// K4 attn_kernel: one CTA = one head x 256 query rows (two 128-row M tiles),
//    384 threads.  Prologue, all warps: the CTA's queries are rotated, given
//    one scale sq = amax / 448 per row and split into three E4M3 pieces
//    (hi + mid + lo, ~12 significant bits) of q / sq, written straight into
//    the swizzled A-operand image in shared memory.  Then:
//   warp 0        loader: one bulk copy per K tile and the scale vectors per
//                 128-slot KV tile, double-buffered (mbarrier + complete_tx)
//   warp 1        MMA issuer (one lane) and TMEM owner (512 columns)
//   warps 2..5    softmax group 0 (rows 0..127; one row per thread / TMEM lane)
//   warps 6..9    softmax group 1 (rows 128..255)
//   warps 10..11  converter: Vt E4M3 tile (read from global memory half a
//                 tile ahead) -> fp16 tile (exact), 128-byte swizzle, two buffers
// Per KV tile j and M tile i:
//   S_i = Q_i K_j^T on tcgen05 kind::f8f6f4: the three Q pieces accumulate into
//         one fp32 TMEM tile, so the score error stays inside the tolerance.
//   softmax: score = S * sq_row * sk_slot * log2(e)/sqrt(D); online max and sum
//         in registers (packed fp32x2 arithmetic, lazy rescaling of O);
//         P = exp2(score - max) * sv_slot / max(sv) -> fp16, written back over
//         S in TMEM.  Three paths by the tile's write groups (the host marks
//         them per tile): one group (one K and one V scale, all in
//         registers), two runs [0, b) and [b, 128) (a write's run of slots
//         ends inside the tile; two scale pairs, all in registers), anything
//         else (per-column scales and validity, out of line: rare on a full
//         ring).
//   O_i += P_i V_j on tcgen05 kind::f16 with P read from TMEM (A operand) and
//         the converted V tile from shared memory (B operand).
// Two M tiles ping-pong so the tensor pipe works on one tile while the other
// is in softmax.  Output: out = O / sum(P''), fp32.
#include <type_traits>

#include "rc_device.cuh"
#include "rc_internal.h"

namespace rc {

// 12 warps: each of the four schedulers of an SM runs one softmax warp of
// each M tile and one of {loader, MMA, converter, converter}, and the
// register file allows 168 registers a thread.
constexpr int kAttnWarps = 12;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kQPieces = 3;
constexpr int kStages = 2;
constexpr int kMTile = 128;
constexpr int kRowsPerCta = 2 * kMTile;
constexpr int kWarpLoad = 0, kWarpMma = 1, kWarpSm0 = 2, kWarpCvt = 10, kCvtWarps = 2;
constexpr uint32_t kTmemCols = 512;
// The converted V tile holds each code's value exactly in fp16 (every finite
// E4M3 value is an fp16 value), so O accumulates P V as is.

// mbarrier indices
enum : int {
    B_KV_FULL = 0,     // [kStages] K tile and scales landed
    B_KV_EMPTY = 2,    // [kStages] the MMA warp and the 8 softmax warps are done with the stage
    B_V16_FULL = 4,    // [2] the converter warps filled the fp16 V buffer
    B_V16_EMPTY = 6,   // [2] both P.V of a tile read the fp16 V buffer
    B_S_FULL = 8,      // [2] scores of M tile i in TMEM
    B_O_DONE = 10,     // [2]
    B_DRAIN = 12,
    B_COUNT = 13
};
static_assert(kStages == 2, "barrier layout assumes two K stages");
// Named (hardware) barriers.  The MMA warp takes each P tile through a
// rendezvous (bar.sync on both sides) instead of polling an mbarrier: the QK
// MMA's operand reads fill the shared-memory pipe, so an mbarrier poll then
// costs ~300 cycles, long enough for the tensor pipe to run dry behind a thread
// whose issue is paced by the MMAs it queues.  Both sides block, so neither can
// run a phase ahead.  The P0 rendezvous of tile t also stands for "fp16 V of
// tile t converted" and "K tile t + 1 landed": one lane of softmax group 0
// tests those mbarriers early in its softmax, so the MMA warp polls nothing.
constexpr int kNbSoftmax = 1;  // the 8 softmax warps (the head's largest V scale)
constexpr int kNbP = 2;        // [2] softmax group of M tile i with the MMA warp: P_i is in TMEM
constexpr int kNbPThreads = 4 * 32 + 32;

template <int D>
struct AttnLayout {
    static constexpr uint32_t kTile = kTileSlots * D;  // bytes of a K tile or a Vt tile
    static constexpr uint32_t kQ = 0;                   // [piece][mtile][128][D] E4M3
    static constexpr uint32_t kQBytes = kQPieces * 2 * kMTile * D;
    static constexpr uint32_t kStage0 = kQBytes;        // K8, sk[128], sv[128], grp[128]
    static constexpr uint32_t kStageBytes = ((kTile + 3 * 512) + 1023) / 1024 * 1024;
    static constexpr uint32_t kV16 = kStage0 + kStages * kStageBytes;  // 2 x [2 halves][D][128 B] fp16
    static constexpr uint32_t kV16One = 2 * D * 128;
    static constexpr uint32_t kV16Bytes = 2 * kV16One;
    static constexpr uint32_t kSq = kV16 + kV16Bytes;  // fp32 [256] row scales
    static constexpr uint32_t kBar = kSq + 2 * kMTile * 4;
    static constexpr uint32_t kMisc = kBar + 8 * B_COUNT;
    static constexpr uint32_t kTotal = kMisc + 64;
    static constexpr uint32_t kAlloc = kTotal + 1024;  // room to align the base to 1024
};

// ---------------------------------------------------------------- K4 attention

// x rounded to 4 significant bits (Veltkamp's splitting with 2^20 + 1 on a
// 24-bit significand): an E4M3 value whenever |x| lies in E4M3's normal
// range, and x - split4(x) is exact.  Plain multiply and subtract, never fused.
__device__ __forceinline__ float split4(float x) {
    const float c = __fmul_rn(x, 1048577.0f);
    return __fsub_rn(c, __fsub_rn(c, x));
}


// Four E4M3 codes (one 32-bit word, code 0 in the low byte) -> four fp16 values,
// exactly, with the hardware conversion (far fewer instructions than placing
// the bits by hand, which matters on the schedulers the softmax warps share).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Softmax of the ring's last tile (fewer than 128 slots) when one write group
// fills it: the uniform arithmetic with the columns past the ring's end cut to
// -inf.  Once a call, so it is kept out of line.  Returns (new running max,
// rescale factor of the old one, the tile's row sum of P'); P goes to TMEM
// columns 0..63.
__device__ __noinline__ float3 last_tile_softmax(uint32_t s_tm, int nvalid, float cu, float lsv0, float lsv,
                                                 float m_run) {
    uint32_t v[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32_async(s_tm + 32 * c, v[c]);
    tmem_wait_ld_dep(v[0]);
    reg_fence(v[1]);
    reg_fence(v[2]);
    reg_fence(v[3]);
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (32 * c + k >= nvalid) v[c][k] = __float_as_uint(-INFINITY);
            mx[k & 3] = fmaxf(mx[k & 3], __uint_as_float(v[c][k]));
        }
    const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * cu;
    const bool bump = (m_run == -INFINITY) || (m_tile > m_run + 8.f);
    const float m_new = bump ? fmaxf(m_run, m_tile) : m_run;
    const float m_fin = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = bump ? ex2(m_run - m_fin) : 1.f;
    const float nmu = lsv0 - (m_fin + lsv);
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
            const float q0 = ex2(fmaf(__uint_as_float(v[c][k]), cu, nmu));
            const float q1 = ex2(fmaf(__uint_as_float(v[c][k + 1]), cu, nmu));
            sum += q0 + q1;
            __half2 h = __floats2half2_rn(q0, q1);
            pk[k / 2] = *reinterpret_cast<uint32_t*>(&h);
        }
        tmem_st16(s_tm + 16 * c, pk);
    }
    return make_float3(m_new, alpha, sum);
}

// Softmax of any other tile (per-column scales, and on a masked tile or one
// the ring ends inside, a validity test): pass A and pass B each read the
// scores from TMEM in 32-column chunks.  Rare on a full ring, so it is kept
// out of line and the hot loop stays small.  Returns (new running max, rescale
// factor of the old one, the tile's row sum); P goes to TMEM columns 0..63.
__device__ __noinline__ float3 general_tile_softmax(uint32_t s_tm, const float* ssk, const float* ssv,
                                                    const int32_t* sgrp, int masked, int nvalid, float a, float lsv,
                                                    float m_run) {
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    // validity of four columns as selects; all of a chunk's scale (and group)
    // loads are issued together, none sits behind a branch
    auto ok4 = [&](int col, bool (&ok)[4]) {
        const int4 g4 = masked ? *reinterpret_cast<const int4*>(sgrp + col) : make_int4(0, 0, 0, 0);
        ok[0] = (col < nvalid) && g4.x >= 0;
        ok[1] = (col + 1 < nvalid) && g4.y >= 0;
        ok[2] = (col + 2 < nvalid) && g4.z >= 0;
        ok[3] = (col + 3 < nvalid) && g4.w >= 0;
    };
    auto max_chunk = [&](const uint32_t (&v)[32], int c) {
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
            const int col = 32 * c + k;
            const float4 s4 = *reinterpret_cast<const float4*>(ssk + col);
            bool ok[4];
            ok4(col, ok);
            const float2 y0 = mul2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), make_float2(s4.x, s4.y));
            const float2 y1 =
                mul2(make_float2(__uint_as_float(v[k + 2]), __uint_as_float(v[k + 3])), make_float2(s4.z, s4.w));
            mx[(k >> 2) & 1] = max3(mx[(k >> 2) & 1], ok[0] ? y0.x : -INFINITY, ok[1] ? y0.y : -INFINITY);
            mx[2 + ((k >> 2) & 1)] = max3(mx[2 + ((k >> 2) & 1)], ok[2] ? y1.x : -INFINITY, ok[3] ? y1.y : -INFINITY);
        }
    };
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(s_tm + 32 * c, v);
        max_chunk(v, c);
    }
    const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a;
    const bool bump = (m_run == -INFINITY) || (m_tile > m_run + 8.f);
    const float m_new = bump ? fmaxf(m_run, m_tile) : m_run;
    const float m_fin = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = bump ? ex2(m_run - m_fin) : 1.f;
    const float msub = m_fin + lsv;
    const float2 a2 = make_float2(a, a), nm2 = make_float2(-msub, -msub);
    float2 ls0 = make_float2(0.f, 0.f), ls1 = make_float2(0.f, 0.f);
    // P' = exp2(S sk a - m - log2(max sv)) * sv; the row sum leaves sv out
    auto p_chunk = [&](const uint32_t (&v)[32], int c) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
            const int col = 32 * c + k;
            const float4 s4 = *reinterpret_cast<const float4*>(ssk + col);
            const float4 v4 = *reinterpret_cast<const float4*>(ssv + col);
            bool ok[4];
            ok4(col, ok);
            const float2 x0 = fma2(mul2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])),
                                        make_float2(s4.x, s4.y)), a2, nm2);
            const float2 x1 = fma2(mul2(make_float2(__uint_as_float(v[k + 2]), __uint_as_float(v[k + 3])),
                                        make_float2(s4.z, s4.w)), a2, nm2);
            const float2 p0 = make_float2(ok[0] ? ex2(x0.x) : 0.f, ok[1] ? ex2(x0.y) : 0.f);
            const float2 p1 = make_float2(ok[2] ? ex2(x1.x) : 0.f, ok[3] ? ex2(x1.y) : 0.f);
            ls0 = add2(ls0, p0);
            ls1 = add2(ls1, p1);
            const float2 q0 = make_float2(ok[0] ? p0.x * v4.x : 0.f, ok[1] ? p0.y * v4.y : 0.f);
            const float2 q1 = make_float2(ok[2] ? p1.x * v4.z : 0.f, ok[3] ? p1.y * v4.w : 0.f);
            __half2 h0 = __floats2half2_rn(q0.x, q0.y);
            __half2 h1 = __floats2half2_rn(q1.x, q1.y);
            pk[k / 2] = *reinterpret_cast<uint32_t*>(&h0);
            pk[k / 2 + 1] = *reinterpret_cast<uint32_t*>(&h1);
        }
        // P chunk c goes to columns 16c..16c+15, which were read in chunks <= c
        tmem_st16(s_tm + 16 * c, pk);
    };
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(s_tm + 32 * c, v);
        p_chunk(v, c);
    }
    return make_float3(m_new, alpha, (ls0.x + ls0.y) + (ls1.x + ls1.y));
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(AttnParams p) {
    using Lay = AttnLayout<D>;
    constexpr uint32_t kSboK = (D == 128) ? 1024u : 512u;  // 8 rows of D bytes
    constexpr uint32_t kSwzK = (D == 128) ? 2u : 4u;       // 128-byte / 64-byte swizzle
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);  // [0] tmem, [2] abort, [4..11] V-scale maxima
    const float* s_sq = reinterpret_cast<const float*>(smem + Lay::kSq);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int row0 = blockIdx.x * kRowsPerCta;
    const int T = p.T;
    AbortState ab{reinterpret_cast<volatile uint32_t*>(&misc[2]), p.status, p.wait_ns};

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[B_KV_FULL + s], 1);
            mbar_init(&bars[B_KV_EMPTY + s], 1 + 8);  // the MMA warp and the 8 softmax warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_V16_FULL + i], kCvtWarps);  // the converter warps
            mbar_init(&bars[B_V16_EMPTY + i], 1);
            mbar_init(&bars[B_S_FULL + i], 1);
            mbar_init(&bars[B_O_DONE + i], 1);
        }
        mbar_init(&bars[B_DRAIN], 1);
        misc[2] = 0u;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&misc[0], kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    auto stage_ptr = [&](int s) { return smem + Lay::kStage0 + s * Lay::kStageBytes; };
    const uint32_t kv_bytes = Lay::kTile + 1024 + (p.masked ? 512 : 0);
    auto load_tile = [&](int j) {
        if (!RC_IN_BOUNDS(j >= 0 && j < T, p.status, kSiteAttnTile)) return;
        const int s = j % kStages;
        uint8_t* st = stage_ptr(s);
        uint64_t* full = &bars[B_KV_FULL + s];
        mbar_arrive_expect_tx(full, kv_bytes);
        bulk_g2s(st, p.kc + (static_cast<size_t>(h) * T + j) * Lay::kTile, Lay::kTile, full);
        bulk_g2s(st + Lay::kTile, p.sk + static_cast<size_t>(h) * p.Cpad + j * kTileSlots, 512, full);
        bulk_g2s(st + Lay::kTile + 512, p.sv + static_cast<size_t>(h) * p.Cpad + j * kTileSlots, 512, full);
        if (p.masked) bulk_g2s(st + Lay::kTile + 1024, p.grp + j * kTileSlots, 512, full);
    };
    // the first KV tiles are on their way while the queries are prepared
    if (warp == kWarpLoad && lane == 0)
        for (int j = 0; j < kStages && j < T; ++j) load_tile(j);

    // ------------------------------------------------------------ query preparation
    // The CTA's bf16 query rows are first copied (cp.async, 16-byte pieces
    // XOR-swizzled by row) into the fp16 V buffers, which the converter fills
    // only after this prologue.  Then each thread takes a quarter of query rows
    // tid/4, tid/4 + 96, ... -- dims 16j + 4q .. 16j + 4q + 3 (q = tid % 4), so
    // that the four threads of a row read its cos/sin in 64 contiguous bytes --
    // with the next row's cos/sin loads in flight while one computes: RoPE at
    // the row's position, one scale sq = amax/448 per row (any scale serves: the
    // softmax multiplies it back), and three E4M3 pieces (hi + mid + lo, ~12
    // significant bits) of q / sq written into the swizzled A-operand image.
    // Rows past n are zero with sq = 1.
    {
        constexpr int DPT = D / 4;                                        // dims per thread
        constexpr int kGroups = DPT / 4;                                  // 4-dim groups per thread
        constexpr int kUnits = D * 2 / 16;                                // 16-byte pieces of a bf16 row
        constexpr int kRowStep = kAttnThreads / 4;                        // rows per pass
        constexpr int kPasses = (kRowsPerCta + kRowStep - 1) / kRowStep;
        uint8_t* qstage = smem + Lay::kV16;                               // [256 rows][D] bf16
        static_assert(kRowsPerCta * D * 2 <= Lay::kV16Bytes, "query rows do not fit the V buffers");
        const int rows_here = min(kRowsPerCta, p.n - row0);
        for (int u = tid; u < rows_here * kUnits; u += kAttnThreads) {
            const int rr = u / kUnits, c = u - rr * kUnits;
            if (!RC_IN_BOUNDS(rr < kRowsPerCta && row0 + rr < p.n, p.status, kSiteAttnQuery)) continue;
            cp_async16(qstage + rr * (D * 2) + ((c ^ (rr & 7)) << 4),
                       p.q + (static_cast<size_t>(row0 + rr) * p.H + h) * D + c * 8);
        }
        const int quarter = tid & 3;
        float* sq_out = reinterpret_cast<float*>(smem + Lay::kSq);
        float4 cs[2][kGroups];  // group j: (cos, sin) of dims 16j + 4q + {0,1} and {2,3}
        auto load_rope = [&](int ps, int buf) {
            const int rr = (tid >> 2) + ps * kRowStep;
            const int row = row0 + rr;
            if (rr < kRowsPerCta && row < p.n) {
                const float4* rsrc = reinterpret_cast<const float4*>(p.rope + static_cast<size_t>(row) * (D / 2));
#pragma unroll
                for (int j = 0; j < kGroups; ++j) cs[buf][j] = __ldg(rsrc + 4 * j + quarter);
            }
        };
        load_rope(0, 0);
        cp_async_wait_all();
        __syncthreads();
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int buf = ps & 1;
            if (ps + 1 < kPasses) load_rope(ps + 1, buf ^ 1);
            const int rr = (tid >> 2) + ps * kRowStep;
            if (rr >= kRowsPerCta) break;  // whole warps leave together
            const int row = row0 + rr;
            float x[DPT];
            float amax = 0.f;
            if (row < p.n) {
#pragma unroll
                for (int j = 0; j < kGroups; ++j) {
                    // dims 16j + 4q .. +3: 8 bytes in piece 2j + q/2 of the row
                    const uint2 qq = *reinterpret_cast<const uint2*>(
                        qstage + rr * (D * 2) + (((2 * j + (quarter >> 1)) ^ (rr & 7)) << 4) + (quarter & 1) * 8);
                    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(&qq);
                    rotate_pair(__bfloat162float(qb[0]), __bfloat162float(qb[1]), cs[buf][j].x, cs[buf][j].y,
                                x[4 * j], x[4 * j + 1]);
                    rotate_pair(__bfloat162float(qb[2]), __bfloat162float(qb[3]), cs[buf][j].z, cs[buf][j].w,
                                x[4 * j + 2], x[4 * j + 3]);
                }
#pragma unroll
                for (int e = 0; e < DPT; ++e) amax = fmaxf(amax, fabsf(x[e]));
            } else {
#pragma unroll
                for (int e = 0; e < DPT; ++e) x[e] = 0.f;
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const float sq = (amax > 0.f) ? amax * (1.f / 448.f) : 1.f;
            const float inv = __fdividef(1.f, sq);
#pragma unroll
            for (int e = 0; e < DPT; ++e) x[e] *= inv;
#pragma unroll
            for (int pc = 0; pc < kQPieces; ++pc) {
                uint8_t* tile = smem + Lay::kQ + (pc * 2 + (rr >> 7)) * (kMTile * D);
#pragma unroll
                for (int j = 0; j < kGroups; ++j) {
                    float y[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // all pieces but the last: x to 4 significant bits (an
                        // E4M3 value), and the exact remainder carries on
                        y[e] = (pc + 1 < kQPieces) ? split4(x[4 * j + e]) : x[4 * j + e];
                        if (pc + 1 < kQPieces) x[4 * j + e] = __fsub_rn(x[4 * j + e], y[e]);
                    }
                    *reinterpret_cast<uint32_t*>(tile + ktile_off(rr & (kMTile - 1), 16 * j + 4 * quarter, D)) =
                        e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
                }
            }
            if (quarter == 0) sq_out[rr] = sq;
        }
        fence_async_smem();  // the tensor core reads the pieces through the async proxy
    }
    __syncthreads();

    if (warp == kWarpLoad) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            // tiles 0 .. kStages-1 went out before the query preparation
            for (int j = kStages; j < T; ++j) {
                const int s = j % kStages;
                if (!mbar_wait(&bars[B_KV_EMPTY + s], ((j / kStages) & 1) ^ 1, ab, kDevTimeoutLoader)) break;
                load_tile(j);
            }
            if (*ab.flag) {
                // leave no copy in flight: wait (bounded) for the last fill of each stage
                for (int s = 0; s < kStages && s < T; ++s) {
                    const int last = ((T - 1 - s) / kStages) * kStages + s;
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(&bars[B_KV_FULL + s], (last / kStages) & 1) &&
                           global_timer_ns() - t0 < 100000000ull) {
                    }
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        // Lane 0 issues; the whole warp takes part in the rendezvous.
        const uint32_t idesc_qk = instr_desc(kFmtE4M3, kFmtE4M3, 128, 128);
        const uint32_t idesc_pv = instr_desc(kFmtF16, kFmtF16, 128, D);
        // Base descriptors, built once: an operand's descriptor differs from its
        // base only in the start-address field (bits 0..13, address / 16), and
        // shared memory ends below 256 KB, so one add moves it without a carry
        // into the other fields.  Issuing an MMA is then two adds and the
        // instruction, which keeps this thread ahead of the tensor pipe while it
        // shares its scheduler with two softmax warps.
        const uint64_t dq0 = smem_desc(smem_u32(smem + Lay::kQ), 16, kSboK, kSwzK);
        const uint64_t dk0 = smem_desc(smem_u32(stage_ptr(0)), 16, kSboK, kSwzK);
        const uint64_t dv0 = smem_desc(smem_u32(smem + Lay::kV16), 16, 1024, 2);
        auto issue_qk = [&](int i, int s) {
            const uint32_t d_tmem = tmem + 128u * i;
            const uint64_t qa = dq0 + static_cast<uint64_t>((i * kMTile * D) >> 4);
            const uint64_t kb = dk0 + static_cast<uint64_t>((s * Lay::kStageBytes) >> 4);
#pragma unroll
            for (int pc = 0; pc < kQPieces; ++pc)
#pragma unroll
                for (int k = 0; k < D / 32; ++k)
                    mma_f8_ss(d_tmem, qa + ((pc * 2 * kMTile * D + k * 32) >> 4), kb + ((k * 32) >> 4), idesc_qk,
                              (pc | k) != 0);
        };
        auto issue_pv = [&](int i, int jt, bool acc) {
            const uint32_t d_tmem = tmem + 256u + static_cast<uint32_t>(D) * i;
            const uint32_t a_tmem = tmem + 128u * i;
            const uint64_t vb = dv0 + static_cast<uint64_t>(((jt & 1) * Lay::kV16One) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_f16_ts(d_tmem, a_tmem + kk * 8, vb + (((kk >> 2) * (D * 128) + (kk & 3) * 32) >> 4), idesc_pv,
                           (acc || kk > 0) ? 1u : 0u);
        };
        // K tile j has landed (lane 0 polls; the warp agrees)
        auto kv_ready = [&](int j) -> bool {
            bool r = true;
            if (lane == 0) r = mbar_wait(&bars[B_KV_FULL + j % kStages], (j / kStages) & 1, ab, kDevTimeoutMma);
            return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
        };
        const bool leader = lane == 0;
        bool ok = kv_ready(0);
        if (ok && leader) {
            tc_fence_after();
            issue_qk(0, 0);
            mma_commit(&bars[B_S_FULL + 0]);
            issue_qk(1, 0);
            mma_commit(&bars[B_S_FULL + 1]);
            mma_commit(&bars[B_KV_EMPTY + 0]);
        }
        // Round j: P.V of tile j - 1 for both M tiles, Q.K of tile j (j < T):
        // PV0(j-1), QK0(j), PV1(j-1), QK1(j).  Every round passes both
        // rendezvous, also after an abort, so no partner is left waiting.
        for (int j = 1; j <= T; ++j) {
            const int s = j % kStages;
            ok = named_barrier_and(kNbP + 0, kNbPThreads, ok);  // P0 and fp16 V of tile j - 1, K tile j
            if (ok && leader) {
                tc_fence_after();
                issue_pv(0, j - 1, j - 1 > 0);
            }
            if (ok && leader) {
                if (j < T) {
                    tc_fence_after();
                    issue_qk(0, s);
                    mma_commit(&bars[B_S_FULL + 0]);
                } else {
                    mma_commit(&bars[B_O_DONE + 0]);
                }
            }
            ok = named_barrier_and(kNbP + 1, kNbPThreads, ok);  // P1 of tile j - 1
            if (ok && leader) {
                tc_fence_after();
                issue_pv(1, j - 1, j - 1 > 0);
                mma_commit(&bars[B_V16_EMPTY + ((j - 1) & 1)]);
                if (j < T) {
                    issue_qk(1, s);
                    mma_commit(&bars[B_S_FULL + 1]);
                    mma_commit(&bars[B_KV_EMPTY + s]);
                } else {
                    mma_commit(&bars[B_O_DONE + 1]);
                }
            }
        }
        if (leader) {
            // every MMA has finished before the tensor memory is released
            mma_commit(&bars[B_DRAIN]);
            uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&bars[B_DRAIN], 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (warp < kWarpCvt) {
        // ------------------------------------------------------------ softmax
        // Row r of M tile mt; scores in log2 units: x = S * sk_col * a with
        // a = sq_row * log2(e)/sqrt(D).  P'' = exp2(x - m - log2(max sv)), so
        // P' = P'' * sv_col = p * sv_col / max sv stays <= 2^8 in fp16 and the
        // shift cancels in out = O / sum(P'').  The running max m only moves
        // (with an O rescale) when a tile raises it by more than 8.
        const int mt = (warp - kWarpSm0) >> 2;    // M tile of this softmax group
        const int quad = warp & 3;                 // TMEM lane quadrant
        const int r = quad * 32 + lane;            // row within the M tile
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t s_tm = tmem + lane_off + 128u * mt;
        const uint32_t o_tm = tmem + lane_off + 256u + static_cast<uint32_t>(D) * mt;
        // the head's largest V scale (empty slots hold 0): the eight softmax warps
        // scan the scales while the first scores are computed
        {
            const float* svh = p.sv + static_cast<size_t>(h) * p.Cpad;
            float m = 0.f;
#pragma unroll 8
            for (int i = tid - kWarpSm0 * 32; i < p.C; i += 256) m = fmaxf(m, svh[i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) reinterpret_cast<float*>(misc)[4 + warp - kWarpSm0] = m;
            named_barrier_sync(kNbSoftmax, 256);
        }
        float svmax = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) svmax = fmaxf(svmax, reinterpret_cast<const float*>(misc)[4 + w]);
        bool ok = true;
        const float a = s_sq[mt * kMTile + r] * p.sm_log2;  // > 0
        const float lsv = (svmax > 0.f) ? lg2_approx(svmax) : 0.f;
        const float2 a2 = make_float2(a, a);
        float m_run = -INFINITY, l_run = 0.f;
        const bool checker = mt == 0 && quad == 0 && lane == 0;  // lane 0 of warp 4
        // softmax of tile j: P into TMEM (over S), O rescaled if the max moved
        auto tile = [&](int j) -> bool {
            const int s = j % kStages;
            // the tile's scales land with its K tile, before its scores: read them first
            if (!warp_wait(&bars[B_KV_FULL + s], (j / kStages) & 1, ab, kDevTimeoutSoftmax)) return false;
            const uint8_t* st = stage_ptr(s);
            const float* ssk = reinterpret_cast<const float*>(st + Lay::kTile);
            const float* ssv = ssk + kTileSlots;
            const int32_t* sgrp = reinterpret_cast<const int32_t*>(ssv + kTileSlots);
            const int nvalid = min(kTileSlots, p.C - j * kTileSlots);
            // one write group fills the tile: one K and one V scale, no per-column loads
            const bool uni = (p.uniform[j >> 6] >> (j & 63)) & 1ull;
            const float cu = uni ? ssk[0] * a : 0.f;
            const float lsv0 = uni ? lg2_approx(ssv[0]) : 0.f;
            const float isv0 = uni ? ex2(-lsv0) : 1.f;
            // a two-run tile needs the scales of its first and last slot only
            const int sb = uni ? 0 : static_cast<int>(p.split[j]);
            const float cuA = ssk[0] * a, cuB = ssk[kTileSlots - 1] * a;
            const float lvA = lg2_approx(ssv[0]), lvB = lg2_approx(ssv[kTileSlots - 1]);
            // Uniform and two-run tiles read nothing more from the stage: release
            // it before the scores arrive, so the loader can refill it a full
            // tile period ahead of its next use.  Other tiles read per-slot
            // scales during their softmax and release the stage after it.
            const bool early_release = uni || sb != 0;
            if (early_release) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_KV_EMPTY + s]);
            }
            // the checker lane: fp16 V of tile j and K tile j + 1 (tested now,
            // the results are read after the softmax, so the shared-memory
            // latency is hidden; a blocking wait follows only if they were late)
            bool vk = true;
            if (checker) {
                vk = mbar_test(&bars[B_V16_FULL + (j & 1)], (j >> 1) & 1);
                if (j + 1 < T) vk = mbar_test(&bars[B_KV_FULL + (j + 1) % kStages], ((j + 1) / kStages) & 1) && vk;
            }
            if (!warp_wait(&bars[B_S_FULL + mt], j & 1, ab, kDevTimeoutSoftmax)) return false;
            tc_fence_after();

            float m_new, alpha;
            float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            // Uniform tile: the row's 128 scores come into registers with four
            // TMEM loads and one wait; pass A (the tile max, one max3 tree) and
            // pass B (the probabilities) both run from the registers.  The ring's
            // last tile (fewer than 128 slots) takes its own instance, so the
            // column cut costs the full tiles nothing.
            auto uniform_tile = [&]() {
                    uint32_t v0[32], v1[32], v2[32], v3[32];
                    tmem_ld32_async(s_tm, v0);
                    tmem_ld32_async(s_tm + 32, v1);
                    tmem_ld32_async(s_tm + 64, v2);
                    tmem_ld32_async(s_tm + 96, v3);
                    tmem_wait_ld_dep(v0);
                    reg_fence(v1);
                    reg_fence(v2);
                    reg_fence(v3);
                    auto chunk_max = [](const uint32_t (&v)[32]) {
                        float t[11];
#pragma unroll
                        for (int i = 0; i < 10; ++i)
                            t[i] = max3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]),
                                        __uint_as_float(v[3 * i + 2]));
                        t[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
                        const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]);
                        const float u2 = max3(t[6], t[7], t[8]), u3 = max3(t[9], t[10], u0);
                        return max3(u1, u2, u3);
                    };
                    const float mxall = fmaxf(fmaxf(chunk_max(v0), chunk_max(v1)), fmaxf(chunk_max(v2), chunk_max(v3)));
                    const float m_tile = mxall * cu;
                    const bool bump = (m_run == -INFINITY) || (m_tile > m_run + 8.f);
                    m_new = bump ? fmaxf(m_run, m_tile) : m_run;
                    const float m_fin = (m_new == -INFINITY) ? 0.f : m_new;
                    alpha = bump ? ex2(m_run - m_fin) : 1.f;
                    const float msub = m_fin + lsv;
                    // P' = exp2(S c - m - log2(max sv) + log2(sv)): the V scale rides in the exponent
                    const float2 cu2 = make_float2(cu, cu);
                    const float2 nmu2 = make_float2(lsv0 - msub, lsv0 - msub);
                    // all four chunks are computed before the stores, so the exp2 work
                    // runs back to back
                    auto p_chunk = [&](const uint32_t (&v)[32], uint32_t* pk) {
#pragma unroll
                        for (int k = 0; k < 32; k += 4) {
                            const float2 x0 = fma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), cu2, nmu2);
                            const float2 x1 =
                                fma2(make_float2(__uint_as_float(v[k + 2]), __uint_as_float(v[k + 3])), cu2, nmu2);
                            const float2 q0 = make_float2(ex2(x0.x), ex2(x0.y));
                            const float2 q1 = make_float2(ex2(x1.x), ex2(x1.y));
                            ls[0] = add2(ls[0], q0);
                            ls[1] = add2(ls[1], q1);
                            __half2 h0 = __floats2half2_rn(q0.x, q0.y);
                            __half2 h1 = __floats2half2_rn(q1.x, q1.y);
                            pk[k / 2] = *reinterpret_cast<uint32_t*>(&h0);
                            pk[k / 2 + 1] = *reinterpret_cast<uint32_t*>(&h1);
                        }
                    };
                    // P (128 slots as 64 fp16 pairs) goes to columns 0..63; the first
                    // half's store is under way while the second half is computed
                    uint32_t pa[32], pb[32];
                    p_chunk(v0, pa);
                    p_chunk(v1, pa + 16);
                    tmem_st32(s_tm, pa);
                    p_chunk(v2, pb);
                    p_chunk(v3, pb + 16);
                    tmem_st32(s_tm + 32, pb);
            };
            // Split tile: slots [0, sb) belong to one write group (scales A) and
            // [sb, 128) to another (B), as where a write's run of slots ends
            // inside a tile.  The 32-column chunk holding column sb is loaded
            // into v3 and the other three into v0..v2, in order: those three run
            // the uniform arithmetic with their chunk's scales, v3 selects A or B
            // per column.  One TMEM round trip, no per-column scale loads.
            auto split_tile = [&](int sb) {
                const int cs = sb >> 5;                   // the chunk holding column sb
                const int eb = sb - 32 * cs;              // its columns in group A: 0..31
                const int c0 = cs > 0 ? 0 : 1, c1 = cs > 1 ? 1 : 2, c2 = cs > 2 ? 2 : 3;
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld32_async(s_tm + 32 * c0, v0);
                tmem_ld32_async(s_tm + 32 * c1, v1);
                tmem_ld32_async(s_tm + 32 * c2, v2);
                tmem_ld32_async(s_tm + 32 * cs, v3);
                tmem_wait_ld_dep(v0);
                reg_fence(v1);
                reg_fence(v2);
                reg_fence(v3);
                auto cmax = [](const uint32_t (&v)[32]) {
                    float t[11];
#pragma unroll
                    for (int i = 0; i < 10; ++i)
                        t[i] = max3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]),
                                    __uint_as_float(v[3 * i + 2]));
                    t[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
                    const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]);
                    const float u2 = max3(t[6], t[7], t[8]), u3 = max3(t[9], t[10], u0);
                    return max3(u1, u2, u3);
                };
                // the scales are positive, so a chunk's max scales with its group's factor
                float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const float x0 = __uint_as_float(v3[k]), x1 = __uint_as_float(v3[k + 1]);
                    mA = max3(mA, k < eb ? x0 : -INFINITY, k + 1 < eb ? x1 : -INFINITY);
                    mB = max3(mB, k < eb ? -INFINITY : x0, k + 1 < eb ? -INFINITY : x1);
                }
                const float m_tile =
                    fmaxf(fmaxf(cmax(v0) * (cs > 0 ? cuA : cuB), cmax(v1) * (cs > 1 ? cuA : cuB)),
                          fmaxf(cmax(v2) * (cs > 2 ? cuA : cuB), fmaxf(mA * cuA, mB * cuB)));
                const bool bump = (m_run == -INFINITY) || (m_tile > m_run + 8.f);
                m_new = bump ? fmaxf(m_run, m_tile) : m_run;
                const float m_fin = (m_new == -INFINITY) ? 0.f : m_new;
                alpha = bump ? ex2(m_run - m_fin) : 1.f;
                const float msub = m_fin + lsv;
                const float nmA = lvA - msub, nmB = lvB - msub;
                const float isvA = ex2(-lvA), isvB = ex2(-lvB);
                // P' = exp2(S c - m - log2(max sv) + log2(sv)); the row sum takes each
                // group's V scale back out
                auto p_one = [&](const uint32_t (&v)[32], int c, bool ga) {
                    const float2 c2 = ga ? make_float2(cuA, cuA) : make_float2(cuB, cuB);
                    const float2 n2 = ga ? make_float2(nmA, nmA) : make_float2(nmB, nmB);
                    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        const float2 x0 = fma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), c2, n2);
                        const float2 x1 =
                            fma2(make_float2(__uint_as_float(v[k + 2]), __uint_as_float(v[k + 3])), c2, n2);
                        const float2 q0 = make_float2(ex2(x0.x), ex2(x0.y));
                        const float2 q1 = make_float2(ex2(x1.x), ex2(x1.y));
                        s0 = add2(s0, q0);
                        s1 = add2(s1, q1);
                        __half2 h0 = __floats2half2_rn(q0.x, q0.y);
                        __half2 h1 = __floats2half2_rn(q1.x, q1.y);
                        pk[k / 2] = *reinterpret_cast<uint32_t*>(&h0);
                        pk[k / 2 + 1] = *reinterpret_cast<uint32_t*>(&h1);
                    }
                    ls[0].x += ((s0.x + s0.y) + (s1.x + s1.y)) * (ga ? isvA : isvB);
                    // P of chunk c goes to columns 16c..16c+15 (every score is in registers)
                    tmem_st16(s_tm + 16 * c, pk);
                };
                p_one(v0, c0, cs > 0);
                p_one(v1, c1, cs > 1);
                p_one(v2, c2, cs > 2);
                {
                    float2 sw = make_float2(0.f, 0.f);
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const bool a0 = k < eb, a1 = k + 1 < eb;
                        const float2 x = fma2(make_float2(__uint_as_float(v3[k]), __uint_as_float(v3[k + 1])),
                                              make_float2(a0 ? cuA : cuB, a1 ? cuA : cuB),
                                              make_float2(a0 ? nmA : nmB, a1 ? nmA : nmB));
                        const float2 q = make_float2(ex2(x.x), ex2(x.y));
                        sw = fma2(q, make_float2(a0 ? isvA : isvB, a1 ? isvA : isvB), sw);
                        __half2 hq = __floats2half2_rn(q.x, q.y);
                        pk[k / 2] = *reinterpret_cast<uint32_t*>(&hq);
                    }
                    ls[0].y += sw.x + sw.y;
                    tmem_st16(s_tm + 16 * cs, pk);
                }
            };
            if (__builtin_expect(uni && nvalid == kTileSlots, 1)) {
                uniform_tile();
            } else if (uni) {
                const float3 r = last_tile_softmax(s_tm, nvalid, cu, lsv0, lsv, m_run);
                m_new = r.x;
                alpha = r.y;
                ls[0].x = r.z;
            } else if (sb != 0) {
                split_tile(sb);
            } else {
                const float3 r = general_tile_softmax(s_tm, ssk, ssv, sgrp, p.masked, nvalid, a, lsv, m_run);
                m_new = r.x;
                alpha = r.y;
                ls[0].x = r.z;
            }
            tmem_st_wait();
            if (!early_release) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_KV_EMPTY + s]);
            }
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
            // on uniform tiles the sum holds P' = P'' * 2^log2(sv): take the V scale back out
            // (split tiles weight their sums per group, with isv0 = 1)
            const float lsum = (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
            l_run = l_run * alpha + lsum * isv0;
            m_run = m_new;
            if (checker && !vk) {
                if (!mbar_wait(&bars[B_V16_FULL + (j & 1)], (j >> 1) & 1, ab, kDevTimeoutSoftmax)) return false;
                if (j + 1 < T &&
                    !mbar_wait(&bars[B_KV_FULL + (j + 1) % kStages], ((j + 1) / kStages) & 1, ab, kDevTimeoutSoftmax))
                    return false;
            }
            return true;
        };
        // every tile passes the P rendezvous with the MMA warp, also after an abort
        for (int j = 0; j < T; ++j) {
            if (ok) ok = tile(j);
            tc_fence_before();
            __syncwarp();
            ok = named_barrier_and(kNbP + mt, kNbPThreads, ok);
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = warp_wait(&bars[B_O_DONE + mt], 0, ab, kDevTimeoutEpilogue);
        if (ok) {
            tc_fence_after();
            const float fin = (l_run > 0.f) ? 1.f / l_run : 0.f;
            // The warp's 32 rows go out through shared memory (the query
            // image, free once both M tiles' last Q.K has finished, which
            // precedes O_DONE on the tensor pipe): each thread parks its row's
            // 32-column chunk, then each store instruction writes 128-byte
            // lines of four rows.  A thread storing its own row would touch 32
            // lines an instruction, a flood that held up the other M tile's
            // TMEM stores by thousands of cycles.
            float* stage = reinterpret_cast<float*>(smem + Lay::kQ) + (warp - kWarpSm0) * (32 * 36);
            const int wrow0 = row0 + mt * kMTile + quad * 32;  // the warp's first query row
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
                    if (wrow0 + r < p.n && RC_IN_BOUNDS(wrow0 + r >= 0, p.status, kSiteAttnOut))
                        *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(wrow0 + r) * p.H + h) * D + 32 * c +
                                                   4 * q) = val;
                }
                __syncwarp();
            }
        }
    } else {
        // ------------------------------------------------------------ V converter
        // Reads each Vt tile straight from global memory (L2: the head's CTAs
        // share it; no L1 allocation, which cost the softmax ~10 % of the
        // kernel) in two halves, each fetched while the one before it is
        // converted, and fills the two fp16 buffers alternately, so it runs
        // ahead of the P.V MMAs.
        constexpr int kCvtThreads = kCvtWarps * 32;
        constexpr int kHalf = D * 8 / kCvtThreads / 2;  // 16-byte units a thread converts per half tile
        const int ct = tid - kWarpCvt * 32;
        uint8_t* v16 = smem + Lay::kV16;
        const uint8_t* vhead = p.vt + static_cast<size_t>(h) * T * Lay::kTile;
        auto fetch = [&](int hh, uint4 (&r)[kHalf]) {
            if (!RC_IN_BOUNDS((hh >> 1) < T, p.status, kSiteAttnVt)) return;
            const uint8_t* src = vhead + static_cast<size_t>(hh >> 1) * Lay::kTile;
#pragma unroll
            for (int k = 0; k < kHalf; ++k)
                r[k] = ldg_nc_na_v4(src + (ct + kCvtThreads * ((hh & 1) * kHalf + k)) * 16);
        };
        bool cok = true;
        // converts half hh of the tile stream; the second half of a tile
        // publishes the buffer
        auto convert = [&](int hh, const uint4 (&r)[kHalf]) {
            const int jt = hh >> 1, b = jt & 1;
            if ((hh & 1) == 0 && cok)
                cok = warp_wait(&bars[B_V16_EMPTY + b], ((jt >> 1) & 1) ^ 1, ab, kDevTimeoutConvert);
            uint8_t* dstb = v16 + b * Lay::kV16One;
#pragma unroll
            for (int k = 0; k < kHalf && cok; ++k) {
                const int u = ct + kCvtThreads * ((hh & 1) * kHalf + k);
                const int rr = u >> 3, cp = u & 7;
                const int c = cp ^ (rr & 7);  // logical 16-slot chunk
                uint32_t o[8];
                e4m3x4_to_f16x4(r[k].x, o[0], o[1]);
                e4m3x4_to_f16x4(r[k].y, o[2], o[3]);
                e4m3x4_to_f16x4(r[k].z, o[4], o[5]);
                e4m3x4_to_f16x4(r[k].w, o[6], o[7]);
                uint8_t* dst = dstb + (c >> 2) * (D * 128) + rr * 128;
                const int l0 = 2 * (c & 3);
                *reinterpret_cast<uint4*>(dst + (((l0) ^ (rr & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(dst + (((l0 + 1) ^ (rr & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
            if ((hh & 1) && cok) {
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_V16_FULL + b]);
            }
        };
        uint4 ra[kHalf], rb[kHalf];
        const int nh = 2 * T;
        if (nh > 0) fetch(0, ra);
        for (int hh = 0; hh < nh; hh += 2) {
            fetch(hh + 1, rb);
            convert(hh, ra);
            if (hh + 2 < nh) fetch(hh + 2, ra);
            convert(hh + 1, rb);
        }
    }

    // ------------------------------------------------------------ teardown
    // a role's other lanes wait here for its lane 0, so every warp arrives at
    // the CTA barrier converged
    __syncwarp();
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
    static std::atomic<uint64_t> configured{0};
    constexpr uint32_t smem = AttnLayout<D>::kAlloc;
    static_assert(smem <= 227 * 1024, "attention shared memory over the sm_103 limit");
    cudaError_t e = smem_limit_once(attn_kernel<D>, smem, configured);
    if (e != cudaSuccess) return e;
    dim3 grid((p.n + kRowsPerCta - 1) / kRowsPerCta, p.H);
    attn_kernel<D><<<grid, kAttnThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_attention(const AttnParams& p, int D, cudaStream_t s) {
    return (D == 128) ? launch_attention_d<128>(p, s) : launch_attention_d<64>(p, s);
}

}  // namespace rc
