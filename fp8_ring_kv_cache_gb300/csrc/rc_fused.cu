// rc_fused.cu -- the write fused into the K/V projection: the single-GPU half
// of the pages' fused FP8 GEMM (paperdot abstract; cpdf.ai blog, "Como rodar
// 57B em tempo real com batch size 1") applied to the step right before the
// cache: the projection's FP8 GEMM writes its K and V straight into the ring
// (RoPE, per-head amax and scale, E4M3 codes), so the bf16 K and V never go
// to HBM and back.
//
// K2f fused_write_kernel: one CTA = one head's K (or V) x 256 tokens (two M
//    tiles of 128); one thread-block cluster spans the blocks of rows of that
//    head and part (up to 8: n <= 2048), so its amax over all n tokens is
//    agreed through DSMEM as in K2.  Two CTAs share an SM (2 d TMEM columns and
//    96 KB of stages each) and a cluster is at most 8 CTAs, which keeps the
//    production write (96 clusters of 3) resident in one wave; a CTA taking
//    both K and V of a head would need clusters of 6, of which only 46 fit.
//    Warp 0 feeds the stages by TMA (tiled, 64-byte swizzle: the two M tiles'
//    X rows, then the head's Wk or Wv rows), warp 1 issues tcgen05.mma
//    kind::f8f6f4 M128 N(d) K32 into TMEM (one accumulator of d columns per M
//    tile), warps 2..5 run the epilogue, one TMEM lane (a token) a thread:
//    pass 1 scales the accumulators (x_scale * w_scale), rotates K by RoPE at
//    the token's position and takes the amax; after the cluster agrees on the
//    head's scale, pass 2 reloads the accumulators, repeats the same fp32
//    arithmetic and stores E4M3 codes into the ring: each token's K row as
//    16-byte chunks into its swizzled K-tile row, or V transposed byte by byte
//    into the Vt tile (a warp's 32 tokens write 32 consecutive slots of one
//    dim row).  The per-element arithmetic after the product is K2's: fp32
//    RoPE with the write's cos/sin table, s = fl32(amax / 448), codes of
//    fl32(x / s) by the same exact division.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "rc_device.cuh"
#include "rc_internal.h"
#include "rc_layout.h"

namespace rc {

constexpr int kFWarps = 6;
constexpr int kFThreads = kFWarps * 32;
constexpr int kFBK = 64;          // bytes (E4M3 elements) of the reduction dimension per stage
constexpr int kFStages = 4;
constexpr int kFRows = 256;       // tokens per CTA (two M tiles)
constexpr int kFWarpLoad = 0, kFWarpMma = 1, kFWarpEpi0 = 2;

enum : int { FB_FULL = 0, FB_EMPTY = kFStages, FB_DONE = 2 * kFStages, FB_DRAIN = FB_DONE + 1, FB_COUNT = FB_DRAIN + 1 };

template <int D>
struct FusedLayout {
    static constexpr uint32_t kA = 128 * kFBK;                // one M tile's X rows of a stage
    static constexpr uint32_t kB = D * kFBK;                  // the head's Wk (or Wv) rows
    static constexpr uint32_t kStage = 2 * kA + kB;           // 24 KB (d = 128) or 20 KB (d = 64)
    static constexpr uint32_t kBar = kFStages * kStage;
    static constexpr uint32_t kMisc = kBar + 8 * FB_COUNT;    // [0] tmem base, [1] abort flag
    static constexpr uint32_t kRed = kMisc + 16;              // float [4]: the epilogue warps' maxima
    static constexpr uint32_t kTab = kRed + 16;               // float [8]: the cluster's maxima
    static constexpr uint32_t kTotal = kTab + 64;
    static constexpr uint32_t kAlloc = kTotal + 1024;
    static constexpr uint32_t kTmemCols = 2 * D;              // two accumulators of d columns
};

// 2-D tiled TMA load of the box at (x = reduction byte offset, y = row) into
// shared memory, completing on bar's transaction count.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

template <int D>
__global__ void __launch_bounds__(kFThreads, 2)
    fused_write_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWk,
                       const __grid_constant__ CUtensorMap tmWv, FusedParams p) {
    using Lay = FusedLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);
    float* red = reinterpret_cast<float*>(smem + Lay::kRed);
    float* tab = reinterpret_cast<float*>(smem + Lay::kTab);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int kv = blockIdx.z;     // 0: K, 1: V
    const int mb = blockIdx.x;     // block of 256 rows = rank in the cluster (the cluster spans blockIdx.x)
    const int nblk = gridDim.x;    // the cluster's size
    const WriteParams& w = p.w;
    const int row0 = mb * kFRows;
    const int nk = p.hidden / kFBK;
    const CUtensorMap* tmW = kv ? &tmWv : &tmWk;
    AbortState ab{reinterpret_cast<volatile uint32_t*>(&misc[1]), w.status, p.wait_ns};
    // every CTA of the cluster is running once this barrier phase completes
    cluster_arrive_relaxed();

    if (tid == 0) {
        for (int s = 0; s < kFStages; ++s) {
            mbar_init(&bars[FB_FULL + s], 1);
            mbar_init(&bars[FB_EMPTY + s], 1);
        }
        mbar_init(&bars[FB_DONE], 1);
        mbar_init(&bars[FB_DRAIN], 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == kFWarpMma) {
        tmem_alloc(&misc[0], Lay::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    auto stage = [&](int s) { return smem + s * Lay::kStage; };

    if (warp == kFWarpLoad) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int k = 0; k < nk; ++k) {
                const int s = k % kFStages;
                if (k >= kFStages &&
                    !mbar_wait(&bars[FB_EMPTY + s], ((k / kFStages) & 1) ^ 1, ab, kDevTimeoutLoader))
                    break;
                uint64_t* full = &bars[FB_FULL + s];
                mbar_arrive_expect_tx(full, Lay::kStage);
                uint8_t* st = stage(s);
                // X rows past n read as zero (out-of-range boxes are filled)
                tma_load_2d(st, &tmX, k * kFBK, row0, full);
                tma_load_2d(st + Lay::kA, &tmX, k * kFBK, row0 + 128, full);
                tma_load_2d(st + 2 * Lay::kA, tmW, k * kFBK, h * D, full);
                issued = k + 1;
            }
            if (*ab.flag) {
                // let the copies in flight land before the CTA exits
                for (int s = 0; s < kFStages && s < issued; ++s) {
                    const int last = ((issued - 1 - s) / kFStages) * kFStages + s;
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(&bars[FB_FULL + s], (last / kFStages) & 1) &&
                           global_timer_ns() - t0 < 100000000ull) {
                    }
                }
            }
        }
    } else if (warp == kFWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc(kFmtE4M3, kFmtE4M3, 128, D);
            // K-major operands with the 64-byte swizzle: 8-row groups 512 bytes
            // apart; a K step of 32 elements is 32 bytes along the row
            const uint64_t d0 = smem_desc(smem_u32(smem), 16, 512, 4);
            bool ok = true;
            for (int k = 0; k < nk; ++k) {
                const int s = k % kFStages;
                ok = mbar_wait(&bars[FB_FULL + s], (k / kFStages) & 1, ab, kDevTimeoutMma);
                if (!ok) break;
                tc_fence_after();
                const uint64_t sd = d0 + static_cast<uint64_t>((s * Lay::kStage) >> 4);
#pragma unroll
                for (int kk = 0; kk < kFBK / 32; ++kk)
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
                        mma_f8_ss(tmem + mt * D, sd + ((mt * Lay::kA + kk * 32) >> 4),
                                  sd + ((2 * Lay::kA + kk * 32) >> 4), idesc, (k | kk) != 0 ? 1u : 0u);
                mma_commit(&bars[FB_EMPTY + s]);
            }
            if (ok) mma_commit(&bars[FB_DONE]);
            // every MMA issued has finished before the tensor memory is released
            mma_commit(&bars[FB_DRAIN]);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&bars[FB_DRAIN], 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
    // the producer's and the issuer's other lanes wait here for lane 0: every
    // warp arrives at the barriers below converged
    __syncwarp();

    // ------------------------------------------------------------ epilogue
    const bool epi = warp >= kFWarpEpi0;
    const int quad = warp & 3;  // TMEM lane quadrant of this warp
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    auto slot_of = [&](int t) -> int {
        if (w.pos == nullptr) {
            const int s = w.slot0 + t;  // t < n <= C
            return s >= w.C ? s - w.C : s;
        }
        return static_cast<int>(floormod64(w.pos[t] - w.delta_total, w.C));
    };
    // columns [32c, 32c + 32) of M tile mt for token t (this thread's TMEM
    // lane): the accumulator times its scale product, and for K rotated at the
    // token's position (fp32, K2's cos/sin)
    const float mul = kv ? p.v_mul : p.k_mul;
    auto chunk = [&](int mt, int c, int t, float (&x)[32]) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + static_cast<uint32_t>(mt * D + 32 * c), v);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __fmul_rn(__uint_as_float(v[e]), mul);
        if (kv == 0 && t < w.n) {
            const float4* cs = reinterpret_cast<const float4*>(w.rope + static_cast<size_t>(t) * (D / 2) + 16 * c);
#pragma unroll
            for (int q = 0; q < 8; ++q) {  // pairs 2q and 2q + 1 of the chunk
                const float4 c4 = __ldg(cs + q);
                float a0, b0, a1, b1;
                rotate_pair(x[4 * q], x[4 * q + 1], c4.x, c4.y, a0, b0);
                rotate_pair(x[4 * q + 2], x[4 * q + 3], c4.z, c4.w, a1, b1);
                x[4 * q] = a0, x[4 * q + 1] = b0, x[4 * q + 2] = a1, x[4 * q + 3] = b1;
            }
        }
    };
    bool eok = true;
    if (epi) {
        // ---- pass 1: the amax over this CTA's tokens
        float am = 0.f;
        eok = warp_wait(&bars[FB_DONE], 0, ab, kDevTimeoutEpilogue);
        if (eok) {
            tc_fence_after();
#pragma unroll 1
            for (int mt = 0; mt < 2; ++mt) {
                const int t = row0 + mt * 128 + quad * 32 + lane;  // rows past n hold zeros
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float x[32];
                    chunk(mt, c, t, x);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) am = max3(am, fabsf(x[e]), fabsf(x[e + 1]));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) red[quad] = am;
    }
    __syncthreads();
    // ---- across the cluster: each CTA pushes its maximum into every CTA's
    // table; one barrier makes them visible
    cluster_wait();  // (the arrival at kernel start) every CTA is running
    if (tid < nblk) {
        const float m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        dsmem_st_u32(map_shared(&tab[mb], tid), __float_as_uint(m));
    }
    cluster_sync();  // the pushes are visible; no CTA touches another's shared memory after this
    float mx = 0.f;
    for (int r = 0; r < nblk; ++r) mx = fmaxf(mx, tab[r]);
    const float sc = (mx > 0.f) ? __fdiv_rn(mx, 448.f) : 1.f;
    const float rc = __frcp_rn(sc);
    // fl32(x / s) by div_by_scale's three steps on packed pairs, as in K2
    const float2 r2 = make_float2(rc, rc), ns2 = make_float2(-sc, -sc);
    auto div2 = [&](float2 x) {
        const float2 q0 = mul2(x, r2);
        return fma2(fma2(q0, ns2, x), r2, q0);
    };

    if (epi && eok && !*ab.flag) {
        // ---- pass 2: the same values again, quantised into the ring
        uint8_t* vhead = w.vt + static_cast<size_t>(h) * w.T * (D * kTileSlots);
#pragma unroll 1
        for (int mt = 0; mt < 2; ++mt) {
            const int t = row0 + mt * 128 + quad * 32 + lane;
            const bool valid = t < w.n;
            const int slot = valid ? slot_of(t) : 0;
            uint8_t* krow = w.kc + static_cast<size_t>(h * w.T + (slot >> 7)) * (kTileSlots * D);
            uint8_t* vtile = vhead + static_cast<size_t>(slot >> 7) * (D * kTileSlots);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float x[32];
                chunk(mt, c, t, x);
                uint32_t o[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float2 a = div2(make_float2(x[4 * q], x[4 * q + 1]));
                    const float2 b = div2(make_float2(x[4 * q + 2], x[4 * q + 3]));
                    o[q] = e4m3x2(a.x, a.y) | (e4m3x2(b.x, b.y) << 16);
                }
                if (valid) {
                    if (kv == 0) {
                        // dims 32c .. 32c + 31: two 16-byte chunks of the slot's K-tile row
                        *reinterpret_cast<uint4*>(krow + ktile_off(slot & 127, 32 * c, D)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4*>(krow + ktile_off(slot & 127, 32 * c + 16, D)) =
                            make_uint4(o[4], o[5], o[6], o[7]);
                    } else {
                        // V transposed: dim 32c + e of this slot; the warp's 32
                        // tokens fill consecutive slots of each dim row
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            vtile[vtile_off(32 * c + e, slot & 127)] =
                                static_cast<uint8_t>(o[e >> 2] >> (8 * (e & 3)));
                    }
                }
            }
            if (valid) {
                (kv ? w.sv : w.sk)[static_cast<size_t>(h) * w.Cpad + slot] = sc;
                if (kv == 0 && h == 0) w.grp[slot] = w.group;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kFWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link against the driver library)
static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load();
    if (f == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        fn.store(f);
    }
    return f;
}

// [rows][inner] bytes, row stride `inner`, boxes of kFBK bytes x box_rows rows,
// 64-byte swizzle, out-of-range elements read as zero
static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kFBK), box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static cudaError_t launch_fused_d(const FusedParams& p, const uint8_t* X, const uint8_t* Wk, const uint8_t* Wv,
                                  cudaStream_t s) {
    CUtensorMap mx, mk, mv;
    const uint64_t F = static_cast<uint64_t>(p.w.H) * D;
    if (!make_map(&mx, X, p.hidden, p.w.n, 128) || !make_map(&mk, Wk, p.hidden, F, D) ||
        !make_map(&mv, Wv, p.hidden, F, D))
        return cudaErrorInvalidValue;
    static std::atomic<uint64_t> configured{0};
    constexpr uint32_t smem = FusedLayout<D>::kAlloc;
    static_assert(smem <= 227 * 1024, "fused write shared memory over the sm_103 limit");
    cudaError_t e = smem_limit_once(fused_write_kernel<D>, smem, configured);
    if (e != cudaSuccess) return e;
    const int nblk = (p.w.n + kFRows - 1) / kFRows;  // <= 8: one portable cluster along the rows
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(nblk, p.w.H, 2);  // z: K, V
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nblk;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_write_kernel<D>, mx, mk, mv, p);
}

cudaError_t launch_fused_write(const FusedParams& p, const uint8_t* X, const uint8_t* Wk, const uint8_t* Wv, int D,
                               cudaStream_t s) {
    return (D == 128) ? launch_fused_d<128>(p, X, Wk, Wv, s) : launch_fused_d<64>(p, X, Wk, Wv, s);
}

}  // namespace rc
