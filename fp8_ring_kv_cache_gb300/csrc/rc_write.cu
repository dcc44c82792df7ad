// rc_write.cu -- the write path (paperdot abstract: "RoPE and FP8 quantization
// applied once per write"; cpdf.ai "Como rodar 57B em tempo real com batch
// size 1": the work moves from read time to write time).
//
// K1 rope_table_kernel: cos/sin of p * theta_i for the n positions of a write,
//    angle formed in fp64 so large positions keep full accuracy.
// K2 write_kernel: one thread-block cluster of 8 CTAs per head.  Each CTA
//    loads its share of the n tokens (bf16 K and V), rotates K, and reduces the
//    head's amax for K and for V across the cluster through distributed
//    shared memory; then every element becomes the E4M3 code of fl32(x / s)
//    with s = fl32(amax / 448) and is scattered into its ring slot: K rows into
//    the swizzled K tile, V through a shared-memory transpose into the Vt tile.
//    HBM traffic is one read of K and V and one write of the codes.
#include "rc_device.cuh"
#include "rc_internal.h"

namespace rc {

__global__ void rope_table_kernel(RopeTableParams p) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= p.n * p.half) return;
    const int t = idx / p.half;
    const int i = idx - t * p.half;
    const int64_t pos = p.pos ? p.pos[t] : p.p0 + t;
    const double ang = static_cast<double>(pos) * p.theta[i];
    double s, c;
    sincos(ang, &s, &c);
    p.table[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
}

cudaError_t launch_rope_table(const RopeTableParams& p, cudaStream_t s) {
    const int total = p.n * p.half;
    rope_table_kernel<<<(total + 255) / 256, 256, 0, s>>>(p);
    return cudaGetLastError();
}

constexpr int kWriteCluster = 8;
constexpr int kWriteWarps = 8;
constexpr int kWriteThreads = kWriteWarps * 32;
constexpr int kWriteTPW = 12;  // tokens per warp per batch
constexpr int kWriteBatch = kWriteWarps * kWriteTPW;

template <int D>
__global__ void __cluster_dims__(kWriteCluster, 1, 1) __launch_bounds__(kWriteThreads)
    write_kernel(WriteParams p) {
    constexpr int EPL = D / 32;       // elements per lane (4 or 2)
    constexpr int HALF = D / 2;
    constexpr int VROW = D + 4;       // padded staging row (bank spread)
    __shared__ __align__(16) uint8_t vstage[kWriteBatch * VROW];
    __shared__ float red[2][kWriteWarps];
    __shared__ float cta_amax[2];
    __shared__ float scales[2];

    const int h = blockIdx.y;
    const int crank = blockIdx.x;     // the cluster spans blockIdx.x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tpc = (p.n + kWriteCluster - 1) / kWriteCluster;
    const int t0 = min(p.n, crank * tpc);
    const int t1 = min(p.n, t0 + tpc);
    const int nbatch = (t1 - t0 + kWriteBatch - 1) / kWriteBatch;
    const int dim0 = lane * EPL;

    float kreg[kWriteTPW][EPL];
    float vreg[kWriteTPW][EPL];

    auto load_batch = [&](int b, bool first_pass, float& amk, float& amv) {
#pragma unroll
        for (int i = 0; i < kWriteTPW; ++i) {
            const int t = t0 + b * kWriteBatch + i * kWriteWarps + warp;
            if (t < t1) {
                const size_t src = (static_cast<size_t>(t) * p.H + h) * D + dim0;
                __nv_bfloat16 kb[EPL], vb[EPL];
                if constexpr (EPL == 4) {
                    *reinterpret_cast<uint2*>(kb) = *reinterpret_cast<const uint2*>(p.K + src);
                    *reinterpret_cast<uint2*>(vb) = *reinterpret_cast<const uint2*>(p.V + src);
                } else {
                    *reinterpret_cast<uint32_t*>(kb) = *reinterpret_cast<const uint32_t*>(p.K + src);
                    *reinterpret_cast<uint32_t*>(vb) = *reinterpret_cast<const uint32_t*>(p.V + src);
                }
                float2 cs[EPL / 2];
#pragma unroll
                for (int j = 0; j < EPL / 2; ++j) cs[j] = p.rope[static_cast<size_t>(t) * HALF + dim0 / 2 + j];
#pragma unroll
                for (int j = 0; j < EPL / 2; ++j) {
                    rotate_pair(__bfloat162float(kb[2 * j]), __bfloat162float(kb[2 * j + 1]), cs[j].x, cs[j].y,
                                kreg[i][2 * j], kreg[i][2 * j + 1]);
                }
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    vreg[i][e] = __bfloat162float(vb[e]);
                    amk = fmaxf(amk, fabsf(kreg[i][e]));
                    amv = fmaxf(amv, fabsf(vreg[i][e]));
                }
                if (first_pass && p.kraw != nullptr) {
                    // read-time ablation store: the unrotated bf16 row and its angles
                    const int64_t pos = p.pos ? p.pos[t] : p.p0 + t;
                    const int slot = static_cast<int>(floormod64(pos - p.delta_total, p.C));
                    const size_t dst = (static_cast<size_t>(h) * p.Cpad + slot) * D + dim0;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        p.kraw[dst + e] = kb[e];
                        p.vraw[dst + e] = vb[e];
                    }
                    if (h == 0) {
#pragma unroll
                        for (int j = 0; j < EPL / 2; ++j)
                            p.slot_rope[static_cast<size_t>(slot) * HALF + dim0 / 2 + j] = cs[j];
                    }
                }
            }
        }
    };

    // ---- phase 1: per-head amax of rotated K and of V over this CTA's tokens
    float amk = 0.f, amv = 0.f;
    for (int b = 0; b < nbatch; ++b) load_batch(b, true, amk, amv);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        amk = fmaxf(amk, __shfl_xor_sync(0xffffffffu, amk, o));
        amv = fmaxf(amv, __shfl_xor_sync(0xffffffffu, amv, o));
    }
    if (lane == 0) {
        red[0][warp] = amk;
        red[1][warp] = amv;
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        float m = 0.f;
        for (int w = 0; w < kWriteWarps; ++w) m = fmaxf(m, red[threadIdx.x][w]);
        cta_amax[threadIdx.x] = m;
    }
    // ---- across the cluster: every CTA reads the 8 partial maxima
    cluster_sync();
    if (threadIdx.x < 2) {
        float m = 0.f;
        for (uint32_t r = 0; r < kWriteCluster; ++r)
            m = fmaxf(m, __uint_as_float(dsmem_ld_u32(map_shared(&cta_amax[threadIdx.x], r))));
        scales[threadIdx.x] = (m > 0.f) ? __fdiv_rn(m, 448.f) : 1.f;
    }
    cluster_sync();  // no CTA touches another's shared memory after this point
    const float sK = scales[0], sV = scales[1];

    // ---- phase 2: quantise and scatter
    for (int b = 0; b < nbatch; ++b) {
        if (nbatch > 1) {
            float dk = 0.f, dv = 0.f;
            load_batch(b, false, dk, dv);
        }
        const int tb = t0 + b * kWriteBatch;
        const int cnt = min(kWriteBatch, t1 - tb);
#pragma unroll
        for (int i = 0; i < kWriteTPW; ++i) {
            const int tl = i * kWriteWarps + warp;
            const int t = tb + tl;
            if (tl < cnt) {
                const int64_t pos = p.pos ? p.pos[t] : p.p0 + t;
                const int slot = static_cast<int>(floormod64(pos - p.delta_total, p.C));
                const int tile = slot >> 7, row = slot & 127;
                uint8_t* krow = p.kc + static_cast<size_t>(h * p.T + tile) * (kTileSlots * D);
                if constexpr (EPL == 4) {
                    const uint32_t lo = e4m3x2(__fdiv_rn(kreg[i][0], sK), __fdiv_rn(kreg[i][1], sK));
                    const uint32_t hi = e4m3x2(__fdiv_rn(kreg[i][2], sK), __fdiv_rn(kreg[i][3], sK));
                    *reinterpret_cast<uint32_t*>(krow + ktile_off(row, dim0, D)) = lo | (hi << 16);
                    const uint32_t vlo = e4m3x2(__fdiv_rn(vreg[i][0], sV), __fdiv_rn(vreg[i][1], sV));
                    const uint32_t vhi = e4m3x2(__fdiv_rn(vreg[i][2], sV), __fdiv_rn(vreg[i][3], sV));
                    *reinterpret_cast<uint32_t*>(vstage + tl * VROW + dim0) = vlo | (vhi << 16);
                } else {
                    const uint32_t k2 = e4m3x2(__fdiv_rn(kreg[i][0], sK), __fdiv_rn(kreg[i][1], sK));
                    *reinterpret_cast<uint16_t*>(krow + ktile_off(row, dim0, D)) = static_cast<uint16_t>(k2);
                    const uint32_t v2 = e4m3x2(__fdiv_rn(vreg[i][0], sV), __fdiv_rn(vreg[i][1], sV));
                    *reinterpret_cast<uint16_t*>(vstage + tl * VROW + dim0) = static_cast<uint16_t>(v2);
                }
                if (lane == 0) {
                    p.sk[static_cast<size_t>(h) * p.Cpad + slot] = sK;
                    p.sv[static_cast<size_t>(h) * p.Cpad + slot] = sV;
                    if (h == 0) p.grp[slot] = p.group;
                }
            }
        }
        __syncthreads();
        // V transposed: consecutive threads take consecutive tokens of one dim row
        for (int idx = threadIdx.x; idx < D * cnt; idx += kWriteThreads) {
            const int d = idx / cnt;
            const int tl = idx - d * cnt;
            const int t = tb + tl;
            const int64_t pos = p.pos ? p.pos[t] : p.p0 + t;
            const int slot = static_cast<int>(floormod64(pos - p.delta_total, p.C));
            uint8_t* vtile = p.vt + static_cast<size_t>(h * p.T + (slot >> 7)) * (D * kTileSlots);
            vtile[vtile_off(d, slot & 127)] = vstage[tl * VROW + d];
        }
        __syncthreads();
    }
}

cudaError_t launch_write(const WriteParams& p, int D, cudaStream_t s) {
    dim3 grid(kWriteCluster, p.H);
    if (D == 128)
        write_kernel<128><<<grid, kWriteThreads, 0, s>>>(p);
    else
        write_kernel<64><<<grid, kWriteThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace rc
