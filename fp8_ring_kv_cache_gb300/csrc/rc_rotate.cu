// rc_rotate.cu -- whole-ring requantisation kernels.
//
// K3 rotate_kernel (paperdot abstract: a reset of the positions rotates the
//    stored keys by the difference): every stored key moves from position p to
//    p + delta in place.
//    One cluster of 8 CTAs per (layer, head); each thread owns one 16-byte
//    chunk (16 codes) of its rows, dequantises and rotates it by delta, and
//    keeps a running amax per write group that it flushes into a shared-memory
//    table when the group changes; the cluster merges the tables through
//    distributed shared memory; then every row is requantised with its group's
//    new scale s = fl32(amax / 448) and written back.  The second pass re-reads
//    the codes the CTA has just read (an L2 hit), so HBM sees one read and one
//    write of the K codes; V is not touched.
// K5 readtime_kernel (the original read-time design the abstract and the
//    cpdf.ai section "Como rodar 57B em tempo real com batch size 1" describe):
//    rebuilds one layer's FP8 ring from the unrotated bf16 store -- RoPE at each
//    slot's CURRENT position (the angle table of the call is built just before
//    by K1 from the device copy of the slots' positions, which every delta
//    moves), one amax per head for K and for V over the whole cache,
//    quantisation -- into a scratch ring that the attention kernel then reads.
#include "rc_device.cuh"
#include "rc_internal.h"

namespace rc {

constexpr int kRotCluster = 8;
constexpr int kRotWarps = 8;
constexpr int kRotThreads = kRotWarps * 32;

// EPL consecutive codes of one row -> fp32 (exact), EPL = 4 or 2.
template <int EPL>
__device__ __forceinline__ void decode_codes(uint32_t packed, float (&y)[EPL]) {
    const float2 a = e4m3x2_to_float2(static_cast<uint16_t>(packed & 0xFFFFu));
    y[0] = a.x;
    y[1] = a.y;
    if constexpr (EPL == 4) {
        const float2 b = e4m3x2_to_float2(static_cast<uint16_t>(packed >> 16));
        y[2] = b.x;
        y[3] = b.y;
    }
}

template <int EPL>
__device__ __forceinline__ uint32_t load_codes(const uint8_t* p) {
    if constexpr (EPL == 4)
        return *reinterpret_cast<const uint32_t*>(p);
    else
        return *reinterpret_cast<const uint16_t*>(p);
}

template <int EPL>
__device__ __forceinline__ void store_codes(uint8_t* p, uint32_t v) {
    if constexpr (EPL == 4)
        *reinterpret_cast<uint32_t*>(p) = v;
    else
        *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(v);
}

template <int EPL>
__device__ __forceinline__ uint32_t encode_codes(const float (&q)[EPL]) {
    uint32_t v = e4m3x2(q[0], q[1]);
    if constexpr (EPL == 4) v |= e4m3x2(q[2], q[3]) << 16;
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// 16 E4M3 codes (one 16-byte chunk) -> 8 (x, y) pairs in fp32, exact.
__device__ __forceinline__ void decode16(const uint4 raw, float2 (&v)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[2 * q] = e4m3x2_to_float2(static_cast<uint16_t>(w[q] & 0xFFFFu));
        v[2 * q + 1] = e4m3x2_to_float2(static_cast<uint16_t>(w[q] >> 16));
    }
}

// (a, b) -> (a c - b s, a s + b c) in the same rounding order as rotate_pair:
// the (-b s, b c) products are rounded first, then fused into a (c, s).
__device__ __forceinline__ float2 rotate2(float2 ab, float2 cs, float2 sc) {
    return fma2(make_float2(ab.x, ab.x), cs, mul2(make_float2(-ab.y, ab.y), sc));
}

template <int D>
__global__ void __cluster_dims__(kRotCluster, 1, 1) __launch_bounds__(kRotThreads)
    rotate_kernel(RotateParams p, int tpc, int* status) {
    constexpr int CPR = D / 16;                 // 16-byte chunks per row
    constexpr int RPI = kRotThreads / CPR;      // rows per pass of the CTA
    extern __shared__ __align__(16) uint32_t gmax[];  // [Cpad] group amax (fp32 bits)
    (void)status;  // read by the bounds-checked build's index checks

    const int crank = blockIdx.x, h = blockIdx.y, l = blockIdx.z;
    const int tid = threadIdx.x;
    const int chunk = tid % CPR;                // logical chunk: dims 16*chunk .. +15
    const int rsub = tid / CPR;
    const int tile0 = min(p.T, crank * tpc);
    const int ntiles = min(p.T, tile0 + tpc) - tile0;
    const int row0 = tile0 * kTileSlots;
    const int nrows = max(0, min(p.C - row0, ntiles * kTileSlots));
    const size_t lh = static_cast<size_t>(l) * p.H + h;
    uint8_t* gkc = p.kc + (lh * p.T + tile0) * static_cast<size_t>(kTileSlots * D);
    float* gsk = p.sk + lh * p.Cpad + row0;
    const int32_t* ggrp = p.grp + static_cast<size_t>(l) * p.Cpad + row0;

    // (cos, sin) and (sin, cos) of this thread's 8 pairs, read through shared
    // memory: indexing the parameter array per thread would serialise on the
    // constant cache every time the compiler reloads it
    __shared__ float2 s_cs[kMaxHalfDim];
    if (tid < D / 2) s_cs[tid] = p.cs[tid];
    __syncthreads();
    float2 cs[8], sc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        cs[j] = s_cs[chunk * 8 + j];
        sc[j] = make_float2(cs[j].y, cs[j].x);
    }
    auto chunk_addr = [&](int r) {
        return gkc + (r >> 7) * (kTileSlots * D) + ktile_off(r & 127, chunk * 16, D);
    };

    for (int i = tid; i < p.Cpad; i += kRotThreads) gmax[i] = 0u;
    cluster_sync();  // every CTA's table is zero before anyone merges into rank 0

    // ---- phase 1: rotated amax per write group (running max, flushed per group run);
    // four rows per thread are loaded before any is used, to keep loads in flight
    constexpr int kBatch = 4;
    float acc = 0.f, scur = 0.f;
    int gcur = -1;
    for (int rb = rsub; rb < nrows; rb += kBatch * RPI) {
        uint4 raw[kBatch];
        int grow[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = rb + b * RPI;
            grow[b] = (r < nrows) ? ggrp[r] : -1;
            if (grow[b] >= 0 && !RC_IN_BOUNDS(grow[b] < p.Cpad && tile0 + (r >> 7) < p.T, status, kSiteRotGroup))
                grow[b] = -1;
            if (grow[b] >= 0) raw[b] = *reinterpret_cast<const uint4*>(chunk_addr(r));
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int g = grow[b];
            if (g < 0) continue;
            if (g != gcur) {
                if (gcur >= 0) atomicMax(&gmax[gcur], __float_as_uint(acc * scur));
                gcur = g;
                scur = gsk[rb + b * RPI];
                acc = 0.f;
            }
            float2 v[8];
            decode16(raw[b], v);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 x = rotate2(v[j], cs[j], sc[j]);
                acc = max3(acc, fabsf(x.x), fabsf(x.y));
            }
        }
    }
    if (gcur >= 0) atomicMax(&gmax[gcur], __float_as_uint(acc * scur));
    __syncthreads();
    // ---- merge the tables into cluster rank 0 (one push per run of equal groups)
    if (crank != 0) {
        for (int r = tid; r < nrows; r += kRotThreads) {
            const int g = ggrp[r];
            if (g >= 0 && RC_IN_BOUNDS(g < p.Cpad, status, kSiteRotGroup) && (r == 0 || ggrp[r - 1] != g))
                dsmem_max_u32(map_shared(&gmax[g], 0), gmax[g]);
        }
    }
    cluster_sync();
    if (crank != 0) {
        for (int r = tid; r < nrows; r += kRotThreads) {
            const int g = ggrp[r];
            if (g >= 0 && RC_IN_BOUNDS(g < p.Cpad, status, kSiteRotGroup) && (r == 0 || ggrp[r - 1] != g))
                gmax[g] = dsmem_ld_u32(map_shared(&gmax[g], 0));
        }
    }
    cluster_sync();  // rank 0's table is not read after this point
    // ---- phase 2: requantise with the group's new scale and write back (codes re-read from L2)
    for (int rb = rsub; rb < nrows; rb += kBatch * RPI) {
        uint4 raw[kBatch];
        int grow[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = rb + b * RPI;
            grow[b] = (r < nrows) ? ggrp[r] : -1;
            if (grow[b] >= 0 && !RC_IN_BOUNDS(grow[b] < p.Cpad && tile0 + (r >> 7) < p.T && row0 + r < p.Cpad,
                                              status, kSiteRotRow))
                grow[b] = -1;
            if (grow[b] >= 0) raw[b] = *reinterpret_cast<const uint4*>(chunk_addr(r));
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int g = grow[b];
            if (g < 0) continue;
            const int r = rb + b * RPI;
            const float amax = __uint_as_float(gmax[g]);
            const float s_new = (amax > 0.f) ? __fdiv_rn(amax, 448.f) : 1.f;
            const float mult = __fdiv_rn(gsk[r], s_new);
            const float2 m2 = make_float2(mult, mult);
            float2 v[8];
            decode16(raw[b], v);
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 x0 = mul2(rotate2(v[2 * q], cs[2 * q], sc[2 * q]), m2);
                const float2 x1 = mul2(rotate2(v[2 * q + 1], cs[2 * q + 1], sc[2 * q + 1]), m2);
                w[q] = e4m3x2(x0.x, x0.y) | (e4m3x2(x1.x, x1.y) << 16);
            }
            *reinterpret_cast<uint4*>(chunk_addr(r)) = make_uint4(w[0], w[1], w[2], w[3]);
            if (chunk == 0) gsk[r] = s_new;
        }
    }
    // the read-time ablation's copy of each slot's position moves with it
    if (p.slot_pos != nullptr && h == 0) {
        int64_t* spos = p.slot_pos + static_cast<size_t>(l) * p.Cpad + row0;
        for (int r = tid; r < nrows; r += kRotThreads)
            if (ggrp[r] >= 0) spos[r] += p.delta;
    }
}

// ---------------------------------------------------------------- K3, staged
// The rotation of rings whose share per CTA fits shared memory (T <= 48 tiles
// at D = 128, 96 at D = 64: the 5,788-slot ring has 46).  Each CTA of the
// cluster of 8 brings its tiles, with their scales and write groups, into
// shared memory by three bulk copies issued at the start, so HBM sees one read
// and one write of every code and every read is in flight at once.
// Both passes then run from shared memory.  A thread takes one 16-byte chunk
// (16 codes, 8 dimension pairs) of two adjacent slots, so one packed fp32x2
// instruction rotates a dimension pair of both slots.  The per-group amax
// table is spread over the cluster: group g's word lives in CTA g % 8, which
// keeps each CTA's table at Cpad / 8 words and two CTAs on an SM.
constexpr uint64_t kStaggerNs = 4000;  // start spacing of the staged rotation's first wave

template <int D>
struct RotStaged {
    static constexpr int kMaxTiles = (D == 128) ? 6 : 12;  // 96 KB of codes
    static constexpr uint32_t kTile = kTileSlots * D;
    static constexpr uint32_t kCodes = 0;
    static constexpr uint32_t kSk = kMaxTiles * kTile;                    // fp32 [kMaxTiles * 128]
    static constexpr uint32_t kGrp = kSk + kMaxTiles * kTileSlots * 4;    // int32 [kMaxTiles * 128]
    static constexpr uint32_t kBar = kGrp + kMaxTiles * kTileSlots * 4;   // mbarrier: the CTA's copies landed
    static constexpr uint32_t kMisc = kBar + 16;                          // [0] abort flag
    static constexpr uint32_t kTab = kMisc + 16;                          // uint32 [Cpad / 8] group amax bits
    static uint32_t bytes(int Cpad) { return kTab + static_cast<uint32_t>(Cpad / kRotCluster) * 4u; }
};

template <int D>
__global__ void __cluster_dims__(kRotCluster, 1, 1) __launch_bounds__(kRotThreads, 2)
    rotate_staged_kernel(RotateParams p, int tpc, int wave, int* status) {
    using Lay = RotStaged<D>;
    constexpr int CPR = D / 16;              // 16-byte chunks per row
    constexpr int PPP = kRotThreads / CPR;   // row pairs per pass
    constexpr int RPP = 2 * PPP;             // rows per pass (64 at D = 128, 128 at D = 64)
    static_assert(kTileSlots % RPP == 0, "a pass stays inside one tile");
    extern __shared__ __align__(1024) uint8_t sm[];
    uint8_t* codes = sm + Lay::kCodes;
    float* ssk = reinterpret_cast<float*>(sm + Lay::kSk);
    int32_t* sgrp = reinterpret_cast<int32_t*>(sm + Lay::kGrp);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::kBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + Lay::kMisc);
    uint32_t* tab = reinterpret_cast<uint32_t*>(sm + Lay::kTab);

    const int crank = blockIdx.x, h = blockIdx.y, l = blockIdx.z;
    const int tid = threadIdx.x;
    const int q = tid % CPR;                 // chunk: dims 16 q .. 16 q + 15
    const int pr = tid / CPR;                // row pair within a pass
    const int tile0 = min(p.T, crank * tpc);
    const int ntiles = min(p.T, tile0 + tpc) - tile0;
    const int row0 = tile0 * kTileSlots;
    const int nrows = max(0, min(p.C - row0, ntiles * kTileSlots));
    const size_t lh = static_cast<size_t>(l) * p.H + h;
    uint8_t* gkc = p.kc + (lh * p.T + tile0) * static_cast<size_t>(Lay::kTile);
    float* gsk = p.sk + lh * p.Cpad + row0;
    const int32_t* ggrp = p.grp + static_cast<size_t>(l) * p.Cpad + row0;
    AbortState ab{reinterpret_cast<volatile uint32_t*>(&misc[0]), status, p.wait_ns};

    // the CTA's tiles are contiguous, and so are their scales and groups:
    // three bulk copies on one barrier
    const bool copy_ok = RC_IN_BOUNDS(
        ntiles <= Lay::kMaxTiles && tile0 + ntiles <= p.T && row0 + ntiles * kTileSlots <= p.Cpad, status,
        kSiteRotCopy);
    if (tid == 0) {
        misc[0] = 0u;
        mbar_init(&bars[0], 1);
        fence_mbar_init();
        // The first wave's clusters (the `wave` clusters resident at once)
        // would otherwise run their phases in lockstep for the whole launch:
        // every CTA loading at once, then every CTA requantising.  Holding
        // their copies back by 0, 4, 8 or 12 us lets the loads of some
        // clusters overlap the stores of others from then on.
        const int cid = blockIdx.y + blockIdx.z * gridDim.y;
        if (cid < wave) {
            const uint64_t hold = static_cast<uint64_t>(cid & 3) * kStaggerNs;
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < hold) __nanosleep(256);
        }
        if (ntiles > 0 && copy_ok) {
            mbar_arrive_expect_tx(&bars[0], ntiles * (Lay::kTile + 2 * kTileSlots * 4));
            bulk_g2s(codes, gkc, ntiles * Lay::kTile, &bars[0]);
            bulk_g2s(ssk, gsk, ntiles * kTileSlots * 4, &bars[0]);
            bulk_g2s(sgrp, ggrp, ntiles * kTileSlots * 4, &bars[0]);
        }
    }
    // (cos, sin) of delta * theta_i through shared memory: indexing the
    // parameter array per thread would serialise on the constant cache
    __shared__ float2 s_cs[kMaxHalfDim];
    if (tid < D / 2) s_cs[tid] = p.cs[tid];
    for (int i = tid; i < p.Cpad / kRotCluster; i += kRotThreads) tab[i] = 0u;
    cluster_sync();  // every table is zero before any peer merges into it; the barriers are initialised
    // the thread's 8 dimension pairs: (c, c), (-s, -s), (s, s)
    float2 cc[8], ns[8], ss[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 cs = s_cs[q * 8 + j];
        cc[j] = make_float2(cs.x, cs.x);
        ns[j] = make_float2(-cs.y, -cs.y);
        ss[j] = make_float2(cs.y, cs.y);
    }

    // byte offset of this thread's chunk of row r (r even) and of row r + 1:
    // the rows have their own swizzle phases
    auto chunk_off = [&](int r, uint32_t& o0, uint32_t& o1) {
        const uint32_t base = (r >> 7) * Lay::kTile;
        o0 = base + ktile_off(r & 127, q * 16, D);
        o1 = base + ktile_off((r & 127) + 1, q * 16, D);
    };
    // rows r and r + 1 of the CTA -> rotated pairs (x of both rows, y of both rows)
    auto rotate_rows = [&](int r, float2 (&X)[8], float2 (&Y)[8]) {
        uint32_t o0, o1;
        chunk_off(r, o0, o1);
        const uint4 a = *reinterpret_cast<const uint4*>(codes + o0);
        const uint4 b = *reinterpret_cast<const uint4*>(codes + o1);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float2 va = e4m3x2_to_float2(static_cast<uint16_t>(wa[j >> 1] >> (16 * (j & 1))));
            const float2 vb = e4m3x2_to_float2(static_cast<uint16_t>(wb[j >> 1] >> (16 * (j & 1))));
            const float2 x = make_float2(va.x, vb.x), y = make_float2(va.y, vb.y);
            // the rounding order of rotate_pair: the y products first, then fused into x (c, s)
            X[j] = fma2(x, cc[j], mul2(y, ns[j]));
            Y[j] = fma2(x, ss[j], mul2(y, cc[j]));
        }
    };
    static_assert(D == 128 || D == 64, "head_dim 64 or 128");

    bool ok = true;
    // ---- pass 1: rotated amax per write group, a running max flushed per run of rows
    float acc = 0.f, scur = 0.f;
    int gcur = -1;
    auto flush = [&]() {
        if (gcur >= 0) dsmem_max_u32(map_shared(&tab[gcur >> 3], gcur & 7), __float_as_uint(acc * scur));
    };
    if (ntiles > 0) ok = copy_ok && mbar_wait(&bars[0], 0, ab, kDevTimeoutLoader);
    for (int i = 0; i < ntiles && ok; ++i) {
#pragma unroll 1
        for (int rb = i * kTileSlots; rb < (i + 1) * kTileSlots; rb += RPP) {
            const int r = rb + 2 * pr;
            const int g0 = (r < nrows) ? sgrp[r] : -1;
            const int g1 = (r + 1 < nrows) ? sgrp[r + 1] : -1;
            if (g0 < 0 && g1 < 0) continue;
            if (!RC_IN_BOUNDS(g0 < p.Cpad && g1 < p.Cpad, status, kSiteRotGroup)) continue;
            float2 X[8], Y[8];
            rotate_rows(r, X, Y);
            float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f;
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                m0 = max3(m0, fabsf(X[j].x), fabsf(Y[j].x));
                m1 = max3(m1, fabsf(X[j].y), fabsf(Y[j].y));
                m2 = max3(m2, fabsf(X[j + 1].x), fabsf(Y[j + 1].x));
                m3 = max3(m3, fabsf(X[j + 1].y), fabsf(Y[j + 1].y));
            }
            const float mr[2] = {fmaxf(m0, m2), fmaxf(m1, m3)};
            const int gr[2] = {g0, g1};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (gr[k] < 0) continue;
                if (gr[k] != gcur) {
                    flush();
                    gcur = gr[k];
                    scur = ssk[r + k];
                    acc = 0.f;
                }
                acc = fmaxf(acc, mr[k]);
            }
        }
    }
    if (ok) flush();
    __syncwarp();
    cluster_sync();  // every merge has landed
    // ---- each row's new scale s = fl32(amax / 448) (stored) and its factor
    // fl32(s_old / s) (kept in ssk for pass 2): the only reads of the peers'
    // tables, after which this CTA arrives at the exit barrier
    if (ok) {
        for (int r = tid; r < nrows; r += kRotThreads) {
            const int g = sgrp[r];
            if (g < 0) continue;
            if (!RC_IN_BOUNDS(g < p.Cpad && row0 + r < p.Cpad, status, kSiteRotRow)) continue;
            const float amax = __uint_as_float(dsmem_ld_u32(map_shared(&tab[g >> 3], g & 7)));
            const float snew = (amax > 0.f) ? __fdiv_rn(amax, 448.f) : 1.f;
            gsk[r] = snew;
            ssk[r] = __fdiv_rn(ssk[r], snew);
        }
    }
    // the arrival only says "done reading the peers' tables": the reads have
    // completed (their values are used above), and nothing this CTA wrote needs
    // ordering for the peers, so it is relaxed (a release would wait for the
    // scale stores)
    __syncwarp();
    cluster_arrive_relaxed();
    __syncthreads();
    // ---- pass 2: requantise with the group's new scale, in place
    for (int i = 0; i < ntiles && ok; ++i) {
#pragma unroll 1
        for (int rb = i * kTileSlots; rb < (i + 1) * kTileSlots; rb += RPP) {
            const int r = rb + 2 * pr;
            const int g0 = (r < nrows) ? sgrp[r] : -1;
            const int g1 = (r + 1 < nrows) ? sgrp[r + 1] : -1;
            if (g0 < 0 && g1 < 0) continue;
            const float u0 = (g0 >= 0) ? ssk[r] : 0.f, u1 = (g1 >= 0) ? ssk[r + 1] : 0.f;
            float2 X[8], Y[8];
            rotate_rows(r, X, Y);
            const float2 u = make_float2(u0, u1);
            uint32_t wa[4] = {0u, 0u, 0u, 0u}, wb[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 x = mul2(X[j], u), y = mul2(Y[j], u);
                wa[j >> 1] |= e4m3x2(x.x, y.x) << (16 * (j & 1));
                wb[j >> 1] |= e4m3x2(x.y, y.y) << (16 * (j & 1));
            }
            uint32_t o0, o1;
            chunk_off(r, o0, o1);
            if (!RC_IN_BOUNDS(tile0 + ((r + 1) >> 7) < p.T, status, kSiteRotRow)) continue;
            if (g0 >= 0) *reinterpret_cast<uint4*>(gkc + o0) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
            if (g1 >= 0) *reinterpret_cast<uint4*>(gkc + o1) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        }
    }
    // the read-time ablation's copy of each slot's position moves with it
    if (ok && p.slot_pos != nullptr && h == 0) {
        int64_t* spos = p.slot_pos + static_cast<size_t>(l) * p.Cpad + row0;
        for (int r = tid; r < nrows; r += kRotThreads)
            if (sgrp[r] >= 0) spos[r] += p.delta;
    }
    if (!ok && copy_ok && tid == 0 && ntiles > 0) {
        // leave no copy in flight into this CTA's shared memory (bounded)
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars[0], 0) && global_timer_ns() - t0 < 100000000ull) {
        }
    }
    __syncwarp();
    cluster_wait();  // every peer has read this CTA's table
}

// Clusters of the staged kernel resident at once on this device (its largest
// shared-memory size), kept per device; 0 where the query fails.
template <int D>
static int staged_wave(uint32_t smem) {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return 0;
    }
    int n = cached[dev].load(std::memory_order_acquire);
    if (n != 0) return n > 0 ? n : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kRotCluster, 64, 1);
    cfg.blockDim = dim3(kRotThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    if (cudaOccupancyMaxActiveClusters(&n, rotate_staged_kernel<D>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = -1;
    }
    cached[dev].store(n, std::memory_order_release);
    return n > 0 ? n : 0;
}

cudaError_t launch_rotate(const RotateParams& p, int D, int layers, cudaStream_t s, int* status) {
    const int tpc = (p.T + kRotCluster - 1) / kRotCluster;
    dim3 grid(kRotCluster, p.H, layers);
    cudaError_t e;
    if (tpc <= ((D == 128) ? RotStaged<128>::kMaxTiles : RotStaged<64>::kMaxTiles)) {
        static std::atomic<uint64_t> done128{0}, done64{0};
        // the stagger pays off over many waves only: a grid of fewer than
        // four waves starts at once
        const long clusters = static_cast<long>(p.H) * layers;
        if (D == 128) {
            const uint32_t smem = RotStaged<128>::bytes(p.Cpad);
            const uint32_t most = RotStaged<128>::bytes(kRotCluster * RotStaged<128>::kMaxTiles * kTileSlots);
            e = smem_limit_once(rotate_staged_kernel<128>, most, done128);
            if (e != cudaSuccess) return e;
            int wave = staged_wave<128>(most);
            if (clusters < 4L * wave) wave = 0;
            rotate_staged_kernel<128><<<grid, kRotThreads, smem, s>>>(p, tpc, wave, status);
        } else {
            const uint32_t smem = RotStaged<64>::bytes(p.Cpad);
            const uint32_t most = RotStaged<64>::bytes(kRotCluster * RotStaged<64>::kMaxTiles * kTileSlots);
            e = smem_limit_once(rotate_staged_kernel<64>, most, done64);
            if (e != cudaSuccess) return e;
            int wave = staged_wave<64>(most);
            if (clusters < 4L * wave) wave = 0;
            rotate_staged_kernel<64><<<grid, kRotThreads, smem, s>>>(p, tpc, wave, status);
        }
        return cudaGetLastError();
    }
    const size_t smem = static_cast<size_t>(p.Cpad) * 4;
    if (D == 128) {
        e = cudaFuncSetAttribute(rotate_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        rotate_kernel<128><<<grid, kRotThreads, smem, s>>>(p, tpc, status);
    } else {
        e = cudaFuncSetAttribute(rotate_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        rotate_kernel<64><<<grid, kRotThreads, smem, s>>>(p, tpc, status);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- K5 read-time

constexpr int kRtCluster = 8;
constexpr int kRtWarps = 16;
constexpr int kRtThreads = kRtWarps * 32;

template <int D>
__device__ __forceinline__ void rt_load_row(const ReadtimeParams& p, int h, int slot, int dim0, float (&k)[D / 32],
                                            float (&v)[D / 32]) {
    constexpr int EPL = D / 32;
    const size_t src = (static_cast<size_t>(h) * p.Cpad + slot) * D + dim0;
    __nv_bfloat16 kb[EPL], vb[EPL];
    if constexpr (EPL == 4) {
        *reinterpret_cast<uint2*>(kb) = *reinterpret_cast<const uint2*>(p.kraw + src);
        *reinterpret_cast<uint2*>(vb) = *reinterpret_cast<const uint2*>(p.vraw + src);
    } else {
        *reinterpret_cast<uint32_t*>(kb) = *reinterpret_cast<const uint32_t*>(p.kraw + src);
        *reinterpret_cast<uint32_t*>(vb) = *reinterpret_cast<const uint32_t*>(p.vraw + src);
    }
#pragma unroll
    for (int j = 0; j < EPL / 2; ++j) {
        const float2 cs = p.slot_rope[static_cast<size_t>(slot) * (D / 2) + dim0 / 2 + j];
        rotate_pair(__bfloat162float(kb[2 * j]), __bfloat162float(kb[2 * j + 1]), cs.x, cs.y, k[2 * j], k[2 * j + 1]);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = __bfloat162float(vb[e]);
}

// One cluster of 8 CTAs per head.  Phase 1: amax of rotated K and of V over
// every occupied slot of the head (the whole cache); the cluster combines the
// eight partial maxima.  Phase 2: quantise every slot with the head's scale.
template <int D>
__global__ void __cluster_dims__(kRtCluster, 1, 1) __launch_bounds__(kRtThreads, 1)
    readtime_kernel(ReadtimeParams p, int tpc) {
    constexpr int EPL = D / 32;
    constexpr int VROW = D + 16;  // staging row stride (16-byte aligned, spreads banks)
    __shared__ __align__(16) uint8_t vstage[kTileSlots * VROW];
    __shared__ float red[2][kRtWarps];
    __shared__ float cta_amax[2];
    __shared__ float scales[2];

    const int crank = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dim0 = lane * EPL;
    const int tile0 = min(p.T, crank * tpc);
    const int ntiles = min(p.T, tile0 + tpc) - tile0;
    const int row0 = tile0 * kTileSlots;
    const int nrows = max(0, min(p.C - row0, ntiles * kTileSlots));

    // ---- phase 1
    float ak = 0.f, av = 0.f;
    for (int r = warp; r < nrows; r += kRtWarps) {
        if (!RC_IN_BOUNDS(row0 + r < p.Cpad, p.status, kSiteRtRow)) continue;
        if (p.grp[row0 + r] < 0) continue;
        float k[EPL], v[EPL];
        rt_load_row<D>(p, h, row0 + r, dim0, k, v);
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            ak = fmaxf(ak, fabsf(k[e]));
            av = fmaxf(av, fabsf(v[e]));
        }
    }
    ak = warp_max(ak);
    av = warp_max(av);
    if (lane == 0) {
        red[0][warp] = ak;
        red[1][warp] = av;
    }
    __syncthreads();
    if (tid < 2) {
        float m = 0.f;
        for (int w = 0; w < kRtWarps; ++w) m = fmaxf(m, red[tid][w]);
        cta_amax[tid] = m;
    }
    cluster_sync();
    if (tid < 2) {
        float m = 0.f;
        for (uint32_t r = 0; r < kRtCluster; ++r)
            m = fmaxf(m, __uint_as_float(dsmem_ld_u32(map_shared(&cta_amax[tid], r))));
        scales[tid] = (m > 0.f) ? __fdiv_rn(m, 448.f) : 1.f;
    }
    cluster_sync();
    const float skv = scales[0], svv = scales[1];
    // ---- phase 2: quantise tile by tile (K rows direct, V through a transpose)
    for (int t = 0; t < ntiles; ++t) {
        const int tile = tile0 + t;
        uint8_t* ktile = p.kc + (static_cast<size_t>(h) * p.T + tile) * (kTileSlots * D);
        uint8_t* vtile = p.vt + (static_cast<size_t>(h) * p.T + tile) * (kTileSlots * D);
        for (int rr = warp; rr < kTileSlots; rr += kRtWarps) {
            const int slot = tile * kTileSlots + rr;
            if (!RC_IN_BOUNDS(tile < p.T && slot < p.Cpad, p.status, kSiteRtTile)) continue;
            const bool occ = (slot < p.C) && (p.grp[slot] >= 0);
            uint32_t kcode = 0, vcode = 0;
            if (occ) {
                float k[EPL], v[EPL];
                rt_load_row<D>(p, h, slot, dim0, k, v);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    k[e] = __fdiv_rn(k[e], skv);
                    v[e] = __fdiv_rn(v[e], svv);
                }
                kcode = encode_codes<EPL>(k);
                vcode = encode_codes<EPL>(v);
            }
            store_codes<EPL>(ktile + ktile_off(rr, dim0, D), kcode);
            store_codes<EPL>(vstage + rr * VROW + dim0, vcode);
            if (lane == 0) {
                p.sk[static_cast<size_t>(h) * p.Cpad + slot] = occ ? skv : 0.f;
                p.sv[static_cast<size_t>(h) * p.Cpad + slot] = occ ? svv : 0.f;
            }
        }
        __syncthreads();
        for (int u = tid; u < D * 8; u += kRtThreads) {
            const int d = u >> 3, c = u & 7;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                w[q] = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    w[q] |= static_cast<uint32_t>(vstage[(c * 16 + q * 4 + b) * VROW + d]) << (8 * b);
            }
            *reinterpret_cast<uint4*>(vtile + vtile_off(d, c * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
    }
}

cudaError_t launch_readtime(const ReadtimeParams& p, int D, cudaStream_t s) {
    const int tpc = (p.T + kRtCluster - 1) / kRtCluster;
    dim3 grid(kRtCluster, p.H);
    if (D == 128)
        readtime_kernel<128><<<grid, kRtThreads, 0, s>>>(p, tpc);
    else
        readtime_kernel<64><<<grid, kRtThreads, 0, s>>>(p, tpc);
    return cudaGetLastError();
}

}  // namespace rc
