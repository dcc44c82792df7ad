// rc_rotate.cu -- whole-ring requantisation kernels.
//
// K3 rotate_kernel (paperdot abstract: "a delta rotation when positions
//    reset"): every stored key moves from position p to p + delta in place.
//    One cluster of 8 CTAs per (layer, head); each CTA bulk-copies its run of
//    tiles (codes, slot scales, slot groups) into shared memory, dequantises and
//    rotates each row by delta, and reduces the amax of every write group in a
//    shared-memory table; the cluster merges the tables through distributed
//    shared memory; then each row is requantised with its group's new scale
//    s = fl32(amax / 448) and written back.  One read and one write of the K
//    codes; V is not touched.
// K5 readtime_kernel (the original read-time design the abstract and the
//    cpdf.ai section "Como rodar 57B em tempo real com batch size 1" describe):
//    rebuilds one layer's FP8 ring from the unrotated bf16 store -- RoPE at each
//    slot's position, one amax per head for K and for V over the whole cache,
//    quantisation -- into a scratch ring that the attention kernel then reads.
#include "rc_device.cuh"
#include "rc_internal.h"

namespace rc {

constexpr int kRotCluster = 8;
constexpr int kRotWarps = 16;
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

// shared-memory carve-up of the rotate kernel
struct RotSmem {
    uint32_t codes, sk, grp, gmax, bar, total;
};
__host__ __device__ inline RotSmem rot_smem(int tpc, int D, int Cpad) {
    RotSmem s;
    s.codes = 0;
    s.sk = s.codes + tpc * kTileSlots * D;
    s.grp = s.sk + tpc * kTileSlots * 4;
    s.gmax = s.grp + tpc * kTileSlots * 4;
    s.bar = s.gmax + ((Cpad * 4 + 15) / 16) * 16;
    s.total = s.bar + 16;
    return s;
}

template <int D>
__global__ void __cluster_dims__(kRotCluster, 1, 1) __launch_bounds__(kRotThreads, 1)
    rotate_kernel(RotateParams p, int tpc, int* status) {
    constexpr int EPL = D / 32;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint32_t abort_flag;
    const RotSmem L = rot_smem(tpc, D, p.Cpad);
    uint8_t* sc = smem + L.codes;
    float* ssk = reinterpret_cast<float*>(smem + L.sk);
    int32_t* sgrp = reinterpret_cast<int32_t*>(smem + L.grp);
    uint32_t* gmax = reinterpret_cast<uint32_t*>(smem + L.gmax);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);

    const int crank = blockIdx.x, h = blockIdx.y, l = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dim0 = lane * EPL;
    const int tile0 = min(p.T, crank * tpc);
    const int ntiles = min(p.T, tile0 + tpc) - tile0;
    const int nrows = max(0, min(p.C - tile0 * kTileSlots, ntiles * kTileSlots));
    const size_t lh = static_cast<size_t>(l) * p.H + h;
    uint8_t* gkc = p.kc + (lh * p.T + tile0) * static_cast<size_t>(kTileSlots * D);
    float* gsk = p.sk + lh * p.Cpad + static_cast<size_t>(tile0) * kTileSlots;
    const int32_t* ggrp = p.grp + static_cast<size_t>(l) * p.Cpad + static_cast<size_t>(tile0) * kTileSlots;

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < p.Cpad; i += kRotThreads) gmax[i] = 0u;
    __syncthreads();
    if (tid == 0 && ntiles > 0) {
        const uint32_t nb = static_cast<uint32_t>(ntiles) * kTileSlots;
        mbar_arrive_expect_tx(bar, nb * D + nb * 8);
        bulk_g2s(sc, gkc, nb * D, bar);
        bulk_g2s(ssk, gsk, nb * 4, bar);
        bulk_g2s(sgrp, ggrp, nb * 4, bar);
    }
    cluster_sync();  // every CTA's table is zero before anyone merges into rank 0
    AbortState ab{&abort_flag, status};
    bool ok = true;
    if (ntiles > 0) ok = mbar_wait(bar, 0, ab, kDevTimeoutLoader);

    float cs_c[EPL / 2], cs_s[EPL / 2];
#pragma unroll
    for (int j = 0; j < EPL / 2; ++j) {
        cs_c[j] = p.cs[dim0 / 2 + j].x;
        cs_s[j] = p.cs[dim0 / 2 + j].y;
    }

    // ---- phase 1: rotated amax per write group (code space times the slot scale)
    if (ok) {
        for (int r = warp; r < nrows; r += kRotWarps) {
            const int g = sgrp[r];
            if (g < 0) continue;
            float y[EPL];
            decode_codes<EPL>(load_codes<EPL>(sc + (r >> 7) * (kTileSlots * D) + ktile_off(r & 127, dim0, D)), y);
            float am = 0.f;
#pragma unroll
            for (int j = 0; j < EPL / 2; ++j) {
                float a, b;
                rotate_pair(y[2 * j], y[2 * j + 1], cs_c[j], cs_s[j], a, b);
                am = fmaxf(am, fmaxf(fabsf(a), fabsf(b)));
            }
            am = warp_max(am);
            if (lane == 0) atomicMax(&gmax[g], __float_as_uint(am * ssk[r]));
        }
    }
    __syncthreads();
    // ---- merge the tables into cluster rank 0 (one push per run of equal groups)
    if (crank != 0) {
        for (int r = tid; r < nrows; r += kRotThreads) {
            const int g = sgrp[r];
            if (g >= 0 && (r == 0 || sgrp[r - 1] != g)) dsmem_max_u32(map_shared(&gmax[g], 0), gmax[g]);
        }
    }
    cluster_sync();
    if (crank != 0) {
        for (int r = tid; r < nrows; r += kRotThreads) {
            const int g = sgrp[r];
            if (g >= 0 && (r == 0 || sgrp[r - 1] != g)) gmax[g] = dsmem_ld_u32(map_shared(&gmax[g], 0));
        }
    }
    cluster_sync();  // rank 0's table is not read after this point
    // ---- phase 2: requantise with the group's new scale and write back
    if (ok) {
        for (int r = warp; r < nrows; r += kRotWarps) {
            const int g = sgrp[r];
            if (g < 0) continue;
            const float amax = __uint_as_float(gmax[g]);
            const float s_new = (amax > 0.f) ? __fdiv_rn(amax, 448.f) : 1.f;
            const float mult = __fdiv_rn(ssk[r], s_new);
            const uint32_t off = (r >> 7) * (kTileSlots * D) + ktile_off(r & 127, dim0, D);
            float y[EPL], q[EPL];
            decode_codes<EPL>(load_codes<EPL>(sc + off), y);
#pragma unroll
            for (int j = 0; j < EPL / 2; ++j) {
                float a, b;
                rotate_pair(y[2 * j], y[2 * j + 1], cs_c[j], cs_s[j], a, b);
                q[2 * j] = a * mult;
                q[2 * j + 1] = b * mult;
            }
            store_codes<EPL>(gkc + off, encode_codes<EPL>(q));
            if (lane == 0) gsk[r] = s_new;
        }
    }
}

cudaError_t launch_rotate(const RotateParams& p, int D, int layers, cudaStream_t s, int* status) {
    const int tpc = (p.T + kRotCluster - 1) / kRotCluster;
    const RotSmem L = rot_smem(tpc, D, p.Cpad);
    dim3 grid(kRotCluster, p.H, layers);
    cudaError_t e;
    if (D == 128) {
        e = cudaFuncSetAttribute(rotate_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
        if (e != cudaSuccess) return e;
        rotate_kernel<128><<<grid, kRotThreads, L.total, s>>>(p, tpc, status);
    } else {
        e = cudaFuncSetAttribute(rotate_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
        if (e != cudaSuccess) return e;
        rotate_kernel<64><<<grid, kRotThreads, L.total, s>>>(p, tpc, status);
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
