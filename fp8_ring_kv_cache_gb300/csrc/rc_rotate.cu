// rc_rotate.cu -- whole-ring requantisation kernels.
//
// K3 rotate_kernel (paperdot abstract: "a delta rotation when positions
//    reset"): every stored key moves from position p to p + delta in place.
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
    (void)status;

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
            if (g >= 0 && (r == 0 || ggrp[r - 1] != g)) dsmem_max_u32(map_shared(&gmax[g], 0), gmax[g]);
        }
    }
    cluster_sync();
    if (crank != 0) {
        for (int r = tid; r < nrows; r += kRotThreads) {
            const int g = ggrp[r];
            if (g >= 0 && (r == 0 || ggrp[r - 1] != g)) gmax[g] = dsmem_ld_u32(map_shared(&gmax[g], 0));
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

cudaError_t launch_rotate(const RotateParams& p, int D, int layers, cudaStream_t s, int* status) {
    const int tpc = (p.T + kRotCluster - 1) / kRotCluster;
    const size_t smem = static_cast<size_t>(p.Cpad) * 4;
    dim3 grid(kRotCluster, p.H, layers);
    cudaError_t e;
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
