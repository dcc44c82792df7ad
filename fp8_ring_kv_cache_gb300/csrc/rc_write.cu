// rc_write.cu -- the write path (paperdot abstract: keys get RoPE and FP8
// quantisation a single time, as they are written; cpdf.ai "Como rodar 57B em
// tempo real com batch size 1": the work moves from read time to write time).
//
// K1 rope_table_kernel: cos/sin of p * theta_i for the n positions of a write,
//    angle formed in fp64 so large positions keep full accuracy.
// K2 write_kernel: one thread-block cluster of 8 CTAs per head.  Each CTA
//    copies its share of the n tokens (one bf16 K row and V row per token)
//    into shared memory, rotates K, and reduces the head's amax for
//    K and for V across the cluster (each CTA pushes its partial maxima into
//    every CTA's shared table; one cluster barrier); then
//    every element becomes the E4M3 code of fl32(x / s) with
//    s = fl32(amax / 448) and is scattered into its ring slot: K rows into the
//    swizzled K tile, V through a shared-memory transpose into the Vt tile.
//    Rows are staged with 16-byte cp.async copies.
//    HBM traffic is one read of K and V and one write of the codes.
#include "rc_device.cuh"
#include "rc_internal.h"

namespace rc {

__global__ void __launch_bounds__(256) rope_table_kernel(RopeTableParams p) {
    // the frequencies go through shared memory: lanes index different ones,
    // which the parameter bank would serve one address at a time
    __shared__ double th[kMaxHalfDim];
    if (threadIdx.x < p.half) th[threadIdx.x] = p.theta[threadIdx.x];
    __syncthreads();
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= p.n * p.half) return;
    const int t = idx / p.half;
    const int i = idx - t * p.half;
    const int64_t pos = p.pos ? p.pos[t] : p.p0 + t;
    const double ang = static_cast<double>(pos) * th[i];
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
    // A token is taken by CPT lanes, each with 16 of its dims: [8c, 8c + 8) and
    // [D/2 + 8c, D/2 + 8c + 8) for lane chunk c, so the 16-byte shared reads of
    // a token's row are contiguous across its lanes.  A warp takes TPS tokens
    // a step, and the per-token work (slot, tile address, scale stores) is
    // shared by TPS tokens of one instruction.
    constexpr int CPT = D / 16;                         // lanes per token
    constexpr int TPS = 32 / CPT;                       // tokens a warp takes per step
    constexpr int TPB = kWriteWarps * TPS;              // tokens the CTA takes per step
    constexpr int kSteps = (kWriteTB + TPB - 1) / TPB;  // steps per staged batch
    constexpr int HALF = D / 2;
    constexpr uint32_t ROWB = D * 2;  // bytes of one bf16 head row
    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16* kbuf = reinterpret_cast<__nv_bfloat16*>(smem + S::kK);
    __nv_bfloat16* vbuf = reinterpret_cast<__nv_bfloat16*>(smem + S::kV);
    uint8_t* vstage = smem + S::kStage;
    int32_t* sslot = reinterpret_cast<int32_t*>(smem + S::kSlot);
    __shared__ float red[2][kWriteWarps];
    __shared__ float amax_tab[2][kWriteCluster];  // [K / V][cluster rank]: each CTA's partial amax

    const int h = blockIdx.y;
    const int crank = blockIdx.x;     // the cluster spans blockIdx.x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ts = lane / CPT, c = lane % CPT;  // the lane's token within the warp's step, its chunk
    const int tpc = (p.n + kWriteCluster - 1) / kWriteCluster;
    const int t0 = min(p.n, crank * tpc);
    const int t1 = min(p.n, t0 + tpc);
    const int nbatch = (t1 - t0 + kWriteTB - 1) / kWriteTB;
    // every CTA of the cluster is running once this barrier phase completes
    cluster_arrive_relaxed();

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
            const int which = r / kUnits, cc = r - which * kUnits;
            const __nv_bfloat16* src = (which ? p.V : p.K) + (static_cast<size_t>(tb + tl) * p.H + h) * D + cc * 8;
            __nv_bfloat16* dst = (which ? vbuf : kbuf) + tl * D + cc * 8;
            if (RC_IN_BOUNDS(tb + tl >= 0 && tb + tl < p.n && tl < kWriteTB, p.status, kSiteWriteStage))
                cp_async16(dst, src);
        }
        cp_async_wait_all();
        __syncthreads();
    };
    // batch-local token of this lane in step st (the last step may run past cnt)
    auto tok = [&](int st) { return st * TPB + warp * TPS + ts; };
    // (cos, sin) of the lane's 8 dimension pairs for every step of a batch, all
    // loads in flight at once: pairs 4c..4c+3 and D/4 + 4c..D/4 + 4c + 3, two
    // pairs a float4
    auto fetch_rope = [&](int tb, int cnt, float4 (&cs)[kSteps][4]) {
#pragma unroll
        for (int st = 0; st < kSteps; ++st) {
            const int t = tb + min(tok(st), cnt - 1);
            const float4* rr = reinterpret_cast<const float4*>(p.rope + static_cast<size_t>(t) * HALF);
            if (!RC_IN_BOUNDS(t >= 0 && t < p.n, p.status, kSiteWriteRope)) rr = reinterpret_cast<const float4*>(p.rope);
            cs[st][0] = __ldg(rr + 2 * c);
            cs[st][1] = __ldg(rr + 2 * c + 1);
            cs[st][2] = __ldg(rr + D / 8 + 2 * c);
            cs[st][3] = __ldg(rr + D / 8 + 2 * c + 1);
        }
    };
    // the lane's 16 dims of token tl: K rotated at its position, and V; word i
    // of a row piece holds dims (2i, 2i + 1), pair i of the lane
    auto row = [&](int tl, const float4 (&cs)[4], float (&k)[16], float (&v)[16]) {
        const uint8_t* kr = reinterpret_cast<const uint8_t*>(kbuf + tl * D);
        const uint8_t* vr = reinterpret_cast<const uint8_t*>(vbuf + tl * D);
        const uint4 k0 = *reinterpret_cast<const uint4*>(kr + 16 * c);
        const uint4 k1 = *reinterpret_cast<const uint4*>(kr + D + 16 * c);
        const uint4 v0 = *reinterpret_cast<const uint4*>(vr + 16 * c);
        const uint4 v1 = *reinterpret_cast<const uint4*>(vr + D + 16 * c);
        const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float cc = (i & 1) ? cs[i >> 1].z : cs[i >> 1].x;
            const float ss = (i & 1) ? cs[i >> 1].w : cs[i >> 1].y;
            rotate_pair(__uint_as_float(kw[i] << 16), __uint_as_float(kw[i] & 0xFFFF0000u), cc, ss, k[2 * i],
                        k[2 * i + 1]);
            v[2 * i] = __uint_as_float(vw[i] << 16);
            v[2 * i + 1] = __uint_as_float(vw[i] & 0xFFFF0000u);
        }
    };

    // ---- phase 1: per-head amax of rotated K and of V over this CTA's tokens
    float amk = 0.f, amv = 0.f;
    for (int b = 0; b < nbatch; ++b) {
        const int tb = t0 + b * kWriteTB;
        const int cnt = min(kWriteTB, t1 - tb);
        float4 cs[kSteps][4];
        fetch_rope(tb, cnt, cs);
        stage_batch(tb, cnt);
#pragma unroll
        for (int st = 0; st < kSteps; ++st) {
            if (st * TPB + warp * TPS >= cnt) break;  // warp-uniform
            // a lane past the batch's end repeats the last token, which the max
            // already holds: no branch
            const int tl = min(tok(st), cnt - 1);
            float k[16], v[16];
            row(tl, cs[st], k, v);
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                amk = max3(amk, fabsf(k[e]), fabsf(k[e + 1]));
                amv = max3(amv, fabsf(v[e]), fabsf(v[e + 1]));
            }
            if (p.kraw != nullptr && tok(st) < cnt) {
                // read-time ablation store: the unrotated bf16 row and the slot's position
                const int slot = slot_of(tb + tl);
                if (!RC_IN_BOUNDS(slot >= 0 && slot < p.C, p.status, kSiteWriteSlot)) continue;
                uint8_t* kd = reinterpret_cast<uint8_t*>(p.kraw + (static_cast<size_t>(h) * p.Cpad + slot) * D);
                uint8_t* vd = reinterpret_cast<uint8_t*>(p.vraw + (static_cast<size_t>(h) * p.Cpad + slot) * D);
                const uint8_t* kr = reinterpret_cast<const uint8_t*>(kbuf + tl * D);
                const uint8_t* vr = reinterpret_cast<const uint8_t*>(vbuf + tl * D);
                *reinterpret_cast<uint4*>(kd + 16 * c) = *reinterpret_cast<const uint4*>(kr + 16 * c);
                *reinterpret_cast<uint4*>(kd + D + 16 * c) = *reinterpret_cast<const uint4*>(kr + D + 16 * c);
                *reinterpret_cast<uint4*>(vd + 16 * c) = *reinterpret_cast<const uint4*>(vr + 16 * c);
                *reinterpret_cast<uint4*>(vd + D + 16 * c) = *reinterpret_cast<const uint4*>(vr + D + 16 * c);
                if (h == 0 && c == 0) p.slot_pos[slot] = p.pos ? p.pos[tb + tl] : p.p0 + tb + tl;
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
    // ---- across the cluster: each CTA pushes its two maxima into every CTA's
    // table, one barrier makes them visible, and every thread reads its own table
    // phase 2's first angles are on their way while the cluster agrees on the scales
    float4 cs[kSteps][4];
    if (nbatch > 0) fetch_rope(t0, min(kWriteTB, t1 - t0), cs);
    cluster_wait();  // (the arrival at kernel start) every CTA is running
    if (threadIdx.x < 2 * kWriteCluster) {
        const int which = threadIdx.x / kWriteCluster, r = threadIdx.x % kWriteCluster;
        float m = 0.f;
        for (int w = 0; w < kWriteWarps; ++w) m = fmaxf(m, red[which][w]);
        dsmem_st_u32(map_shared(&amax_tab[which][crank], r), __float_as_uint(m));
    }
    cluster_sync();  // the pushes are visible; no CTA touches another's shared memory after this
    float mk = 0.f, mv = 0.f;
#pragma unroll
    for (int r = 0; r < kWriteCluster; ++r) {
        mk = fmaxf(mk, amax_tab[0][r]);
        mv = fmaxf(mv, amax_tab[1][r]);
    }
    const float sK = (mk > 0.f) ? __fdiv_rn(mk, 448.f) : 1.f;
    const float sV = (mv > 0.f) ? __fdiv_rn(mv, 448.f) : 1.f;
    const float rK = __frcp_rn(sK), rV = __frcp_rn(sV);
    // fl32(x / s) by div_by_scale's three steps on packed pairs (fma(q0, -s, x)
    // equals fma(-q0, s, x) exactly)
    const float2 rK2 = make_float2(rK, rK), nsK2 = make_float2(-sK, -sK);
    const float2 rV2 = make_float2(rV, rV), nsV2 = make_float2(-sV, -sV);
    auto div2 = [](float2 x, float2 r, float2 ns) {
        const float2 q0 = mul2(x, r);
        return fma2(fma2(q0, ns, x), r, q0);
    };

    // ---- phase 2: quantise and scatter (a single batch is still staged)
    for (int b = 0; b < nbatch; ++b) {
        const int tb = t0 + b * kWriteTB;
        const int cnt = min(kWriteTB, t1 - tb);
        if (b > 0) fetch_rope(tb, cnt, cs);
        if (nbatch > 1) stage_batch(tb, cnt);
#pragma unroll
        for (int st = 0; st < kSteps; ++st) {
            if (st * TPB + warp * TPS >= cnt) break;  // warp-uniform
            const int tw = tok(st);
            const bool live = tw < cnt;
            const int tl = min(tw, cnt - 1);
            float k[16], v[16];
            row(tl, cs[st], k, v);
            const int slot = slot_of(tb + tl);
            const bool in_range = RC_IN_BOUNDS(slot >= 0 && slot < p.C && tw < kWriteTB, p.status, kSiteWriteSlot);
            uint32_t kq[8], vq[8];  // codes of pairs i (16 bits each)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 a = div2(make_float2(k[2 * i], k[2 * i + 1]), rK2, nsK2);
                const float2 bq = div2(make_float2(v[2 * i], v[2 * i + 1]), rV2, nsV2);
                kq[i] = e4m3x2(a.x, a.y);
                vq[i] = e4m3x2(bq.x, bq.y);
            }
            if (live && in_range) {
                uint8_t* ktile = p.kc + static_cast<size_t>(h * p.T + (slot >> 7)) * (kTileSlots * D);
                *reinterpret_cast<uint2*>(ktile + ktile_off(slot & 127, 8 * c, D)) =
                    make_uint2(kq[0] | (kq[1] << 16), kq[2] | (kq[3] << 16));
                *reinterpret_cast<uint2*>(ktile + ktile_off(slot & 127, HALF + 8 * c, D)) =
                    make_uint2(kq[4] | (kq[5] << 16), kq[6] | (kq[7] << 16));
                *reinterpret_cast<uint2*>(vstage + tw * S::kVRow + 8 * c) =
                    make_uint2(vq[0] | (vq[1] << 16), vq[2] | (vq[3] << 16));
                *reinterpret_cast<uint2*>(vstage + tw * S::kVRow + HALF + 8 * c) =
                    make_uint2(vq[4] | (vq[5] << 16), vq[6] | (vq[7] << 16));
                if (c == 0) {
                    sslot[tw] = slot;
                    p.sk[static_cast<size_t>(h) * p.Cpad + slot] = sK;
                    p.sv[static_cast<size_t>(h) * p.Cpad + slot] = sV;
                    if (h == 0) p.grp[slot] = p.group;
                }
            }
        }
        __syncthreads();
        // V transposed: warp w takes dims [16w', 16w' + 16) (w' = w, w + 8, ...),
        // each lane its tokens; one 16-byte shared load gives a token's 16
        // codes, which go to 16 rows of the token's Vt column
        uint8_t* vhead = p.vt + static_cast<size_t>(h) * p.T * (D * kTileSlots);
        for (int tl = lane; tl < cnt; tl += 32) {
            const int slot = sslot[tl];
            if (!RC_IN_BOUNDS(slot >= 0 && slot < p.C, p.status, kSiteWriteVStage)) continue;
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
    static std::atomic<uint64_t> configured{0};
    constexpr uint32_t smem = WriteSmem<D>::kTotal;
    cudaError_t e = smem_limit_once(write_kernel<D>, smem, configured);
    if (e != cudaSuccess) return e;
    dim3 grid(kWriteCluster, p.H);
    write_kernel<D><<<grid, kWriteThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_write(const WriteParams& p, int D, cudaStream_t s) {
    return (D == 128) ? launch_write_d<128>(p, s) : launch_write_d<64>(p, s);
}

}  // namespace rc
