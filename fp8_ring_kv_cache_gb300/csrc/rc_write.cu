// rc_write.cu -- the write path (paperdot abstract: "RoPE and FP8 quantization
// applied once per write"; cpdf.ai "Como rodar 57B em tempo real com batch
// size 1": the work moves from read time to write time).
//
// K1 rope_table_kernel: cos/sin of p * theta_i for the n positions of a write,
//    angle formed in fp64 so large positions keep full accuracy.
// K2 write_kernel: one thread-block cluster of 8 CTAs per head.  Each CTA
//    copies its share of the n tokens (one bf16 K row and V row per token)
//    into shared memory, rotates K, and reduces the head's amax for
//    K and for V across the cluster through distributed shared memory; then
//    every element becomes the E4M3 code of fl32(x / s) with
//    s = fl32(amax / 448) and is scattered into its ring slot: K rows into the
//    swizzled K tile, V through a shared-memory transpose into the Vt tile.
//    Rows are staged with 16-byte cp.async copies.
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
constexpr int kWriteTB = 96;  // tokens staged in shared memory per batch
constexpr int kWritePer = kWriteTB / kWriteWarps;  // tokens a warp takes per batch

template <int D>
struct WriteSmem {
    static constexpr int kVRow = D + 16;  // V staging row: 16-byte aligned, 16-byte reads of consecutive rows spread over the banks
    static constexpr uint32_t kK = 0;                                   // bf16 [TB][D]
    static constexpr uint32_t kV = kK + kWriteTB * D * 2;               // bf16 [TB][D]
    static constexpr uint32_t kStage = kV + kWriteTB * D * 2;           // u8 [TB][kVRow]
    static constexpr uint32_t kSlot = kStage + kWriteTB * kVRow;        // int32 [TB]
    static constexpr uint32_t kTotal = kSlot + kWriteTB * 4;
};

template <int D>
__global__ void __cluster_dims__(kWriteCluster, 1, 1) __launch_bounds__(kWriteThreads, 3)
    write_kernel(WriteParams p) {
    using S = WriteSmem<D>;
    constexpr int EPL = D / 32;       // elements per lane (4 or 2)
    constexpr int HALF = D / 2;
    constexpr uint32_t ROWB = D * 2;  // bytes of one bf16 head row
    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16* kbuf = reinterpret_cast<__nv_bfloat16*>(smem + S::kK);
    __nv_bfloat16* vbuf = reinterpret_cast<__nv_bfloat16*>(smem + S::kV);
    uint8_t* vstage = smem + S::kStage;
    int32_t* sslot = reinterpret_cast<int32_t*>(smem + S::kSlot);
    __shared__ float red[2][kWriteWarps];
    __shared__ float cta_amax[2];
    __shared__ float scales[2];

    const int h = blockIdx.y;
    const int crank = blockIdx.x;     // the cluster spans blockIdx.x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tpc = (p.n + kWriteCluster - 1) / kWriteCluster;
    const int t0 = min(p.n, crank * tpc);
    const int t1 = min(p.n, t0 + tpc);
    const int nbatch = (t1 - t0 + kWriteTB - 1) / kWriteTB;
    const int dim0 = lane * EPL;

    // slot of token t: floormod(pos - delta_total, C); an arithmetic run starts at slot0
    auto slot_of = [&](int t) -> int {
        if (p.pos == nullptr) {
            const int s = p.slot0 + t;  // t < n <= C
            return s >= p.C ? s - p.C : s;
        }
        return static_cast<int>(floormod64(p.pos[t] - p.delta_total, p.C));
    };
    // bring tokens [tb, tb + cnt) of this head into shared memory: every thread
    // copies 16-byte pieces of the K and V rows with cp.async (many small
    // row-sized bulk copies were several times slower)
    auto stage_batch = [&](int tb, int cnt) {
        constexpr int kUnits = ROWB / 16;  // 16-byte pieces of one row
        const int total = cnt * 2 * kUnits;
        for (int u = threadIdx.x; u < total; u += kWriteThreads) {
            const int tl = u / (2 * kUnits), r = u - tl * (2 * kUnits);
            const int which = r / kUnits, c = r - which * kUnits;
            const __nv_bfloat16* src = (which ? p.V : p.K) + (static_cast<size_t>(tb + tl) * p.H + h) * D + c * 8;
            __nv_bfloat16* dst = (which ? vbuf : kbuf) + tl * D + c * 8;
            cp_async16(dst, src);
        }
        cp_async_wait_all();
        __syncthreads();
    };
    // cos/sin pairs of this lane's dims for the warp's tokens of a batch, all
    // loads in flight at once (one L2 round trip instead of one per token)
    auto fetch_rope = [&](int tb, int cnt, float2 (&cs)[kWritePer][EPL / 2]) {
#pragma unroll
        for (int i = 0; i < kWritePer; ++i) {
            const int tl = warp + kWriteWarps * i;
            const float2* rr = p.rope + static_cast<size_t>(tb + min(tl, cnt - 1)) * HALF + dim0 / 2;
#pragma unroll
            for (int j = 0; j < EPL / 2; ++j) cs[i][j] = __ldg(rr + j);
        }
    };
    // token tl of the staged batch: K rotated at its position (EPL values of this lane) and V
    auto row = [&](int tl, const float2 (&cs)[EPL / 2], float (&k)[EPL], float (&v)[EPL]) {
        __nv_bfloat16 kb[EPL], vb[EPL];
        if constexpr (EPL == 4) {
            *reinterpret_cast<uint2*>(kb) = *reinterpret_cast<const uint2*>(kbuf + tl * D + dim0);
            *reinterpret_cast<uint2*>(vb) = *reinterpret_cast<const uint2*>(vbuf + tl * D + dim0);
        } else {
            *reinterpret_cast<uint32_t*>(kb) = *reinterpret_cast<const uint32_t*>(kbuf + tl * D + dim0);
            *reinterpret_cast<uint32_t*>(vb) = *reinterpret_cast<const uint32_t*>(vbuf + tl * D + dim0);
        }
#pragma unroll
        for (int j = 0; j < EPL / 2; ++j)
            rotate_pair(__bfloat162float(kb[2 * j]), __bfloat162float(kb[2 * j + 1]), cs[j].x, cs[j].y, k[2 * j],
                        k[2 * j + 1]);
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[e] = __bfloat162float(vb[e]);
    };

    // ---- phase 1: per-head amax of rotated K and of V over this CTA's tokens
    float amk = 0.f, amv = 0.f;
    for (int b = 0; b < nbatch; ++b) {
        const int tb = t0 + b * kWriteTB;
        const int cnt = min(kWriteTB, t1 - tb);
        float2 cs[kWritePer][EPL / 2];
        fetch_rope(tb, cnt, cs);
        stage_batch(tb, cnt);
        {
#pragma unroll
            for (int i = 0; i < kWritePer; ++i) {
                const int tl = warp + kWriteWarps * i;
                if (tl >= cnt) break;
                float k[EPL], v[EPL];
                row(tl, cs[i], k, v);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    amk = fmaxf(amk, fabsf(k[e]));
                    amv = fmaxf(amv, fabsf(v[e]));
                }
                if (p.kraw != nullptr) {
                    // read-time ablation store: the unrotated bf16 row and its angles
                    const int slot = slot_of(tb + tl);
                    const size_t dst = (static_cast<size_t>(h) * p.Cpad + slot) * D + dim0;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        p.kraw[dst + e] = kbuf[tl * D + dim0 + e];
                        p.vraw[dst + e] = vbuf[tl * D + dim0 + e];
                    }
                    if (h == 0) {
#pragma unroll
                        for (int j = 0; j < EPL / 2; ++j)
                            p.slot_rope[static_cast<size_t>(slot) * HALF + dim0 / 2 + j] =
                                p.rope[static_cast<size_t>(tb + tl) * HALF + dim0 / 2 + j];
                    }
                }
            }
        }
        __syncthreads();  // the next batch overwrites the staging buffers
    }
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
    const float rK = __frcp_rn(sK), rV = __frcp_rn(sV);

    // ---- phase 2: quantise and scatter (a single batch is still staged)
    for (int b = 0; b < nbatch; ++b) {
        const int tb = t0 + b * kWriteTB;
        const int cnt = min(kWriteTB, t1 - tb);
        float2 cs[kWritePer][EPL / 2];
        fetch_rope(tb, cnt, cs);
        if (nbatch > 1) stage_batch(tb, cnt);
#pragma unroll
        for (int i = 0; i < kWritePer; ++i) {
            const int tl = warp + kWriteWarps * i;
            if (tl >= cnt) break;
            float k[EPL], v[EPL];
            row(tl, cs[i], k, v);
            const int slot = slot_of(tb + tl);
            if (lane == 0) sslot[tl] = slot;
            uint8_t* ktile = p.kc + static_cast<size_t>(h * p.T + (slot >> 7)) * (kTileSlots * D);
            float qk[EPL], qv[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qk[e] = div_by_scale(k[e], sK, rK);
                qv[e] = div_by_scale(v[e], sV, rV);
            }
            if constexpr (EPL == 4) {
                *reinterpret_cast<uint32_t*>(ktile + ktile_off(slot & 127, dim0, D)) =
                    e4m3x2(qk[0], qk[1]) | (e4m3x2(qk[2], qk[3]) << 16);
                *reinterpret_cast<uint32_t*>(vstage + tl * S::kVRow + dim0) =
                    e4m3x2(qv[0], qv[1]) | (e4m3x2(qv[2], qv[3]) << 16);
            } else {
                *reinterpret_cast<uint16_t*>(ktile + ktile_off(slot & 127, dim0, D)) =
                    static_cast<uint16_t>(e4m3x2(qk[0], qk[1]));
                *reinterpret_cast<uint16_t*>(vstage + tl * S::kVRow + dim0) =
                    static_cast<uint16_t>(e4m3x2(qv[0], qv[1]));
            }
            if (lane == 0) {
                p.sk[static_cast<size_t>(h) * p.Cpad + slot] = sK;
                p.sv[static_cast<size_t>(h) * p.Cpad + slot] = sV;
                if (h == 0) p.grp[slot] = p.group;
            }
        }
        __syncthreads();
        // V transposed: warp w takes dims [16w', 16w' + 16) (w' = w, w + 8, ...),
        // each lane its tokens; one 16-byte shared load gives a token's 16
        // codes, which go to 16 rows of the token's Vt column
        uint8_t* vhead = p.vt + static_cast<size_t>(h) * p.T * (D * kTileSlots);
        for (int tl = lane; tl < cnt; tl += 32) {
            const int slot = sslot[tl];
            // Vt byte of (d, slot): tile base + d * 128 + ((chunk ^ (d & 7)) << 4) + (slot & 15)
            uint8_t* base = vhead + static_cast<size_t>(slot >> 7) * (D * kTileSlots) + (slot & 15);
            const int chunk = (slot >> 4) & 7;
            for (int d0 = warp * 16; d0 < D; d0 += kWriteWarps * 16) {
                const uint4 w = *reinterpret_cast<const uint4*>(vstage + tl * S::kVRow + d0);
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    base[(d0 + k) * 128 + ((chunk ^ (k & 7)) << 4)] = static_cast<uint8_t>(words[k >> 2] >> (8 * (k & 3)));
            }
        }
        __syncthreads();
    }
}

template <int D>
static cudaError_t launch_write_d(const WriteParams& p, cudaStream_t s) {
    static bool configured = false;
    constexpr uint32_t smem = WriteSmem<D>::kTotal;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(write_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(kWriteCluster, p.H);
    write_kernel<D><<<grid, kWriteThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_write(const WriteParams& p, int D, cudaStream_t s) {
    return (D == 128) ? launch_write_d<128>(p, s) : launch_write_d<64>(p, s);
}

}  // namespace rc
