// rc_window.cu -- the copy-based window, an ablation of the ring (paperdot
// abstract: the window advances "without copies"; this is the copy that the
// ring avoids).  A cache that concatenates keeps its tokens in position order
// and, when n new positions arrive, moves every stored token n slots down
// before it writes them at the end.  Here that cache is the ring plus a slot
// offset, and the move is K6.
//
// K6 window_shift_kernel: in every layer the slot axis rotates by k -- slot s
// takes what slot (s + k) mod C held -- from one buffer bank into the other:
// K codes in 16-byte pieces of a slot's row, transposed V codes byte by byte
// (a V tile row is slot-minor, so a shift by k moves bytes across its 16-byte
// chunks; the loads are cached, so each source line is fetched once), the
// slots' scales and their write groups.  Padding slots (C .. Cpad) are never
// read; in the V tiles they are written as zero codes, as the rings start.
#include "rc_device.cuh"
#include "rc_internal.h"
#include "rc_layout.h"

namespace rc {

template <int D>
__global__ void __launch_bounds__(256) window_shift_kernel(ShiftParams p) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t LH = static_cast<size_t>(p.L) * p.H;
    const size_t tile = static_cast<size_t>(kTileSlots) * D;  // bytes of one K or V tile
    const size_t ring = static_cast<size_t>(p.T) * tile;     // bytes of one (layer, head) ring
    // 0 <= k < C, so s + k < 2C
    auto src_slot = [&](int s) {
        const int q = s + p.k;
        return q >= p.C ? q - p.C : q;
    };
    if (blockIdx.y == 0) {
        // K: one 16-byte piece (slot s, dims 16c .. 16c + 15) per item
        constexpr int CPR = D / 16;
        const size_t n = LH * static_cast<size_t>(p.C) * CPR;
        for (size_t i = i0; i < n; i += stride) {
            const int c = static_cast<int>(i % CPR);
            const size_t r = i / CPR;
            const int s = static_cast<int>(r % p.C);
            const size_t lh = r / p.C;
            const int q = src_slot(s);
            const uint8_t* src = p.kc_src + lh * ring + static_cast<size_t>(q >> 7) * tile + ktile_off(q & 127, 16 * c, D);
            uint8_t* dst = p.kc_dst + lh * ring + static_cast<size_t>(s >> 7) * tile + ktile_off(s & 127, 16 * c, D);
            *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
        }
    } else if (blockIdx.y == 1) {
        // V: one 16-slot piece of one dim row per item, gathered byte by byte
        const int units = p.Cpad / 16;
        const size_t n = LH * D * static_cast<size_t>(units);
        for (size_t i = i0; i < n; i += stride) {
            const int u = static_cast<int>(i % units);
            const size_t r = i / units;
            const int d = static_cast<int>(r % D);
            const size_t lh = r / D;
            const uint8_t* vsrc = p.vt_src + lh * ring;
            const int s0 = 16 * u;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int s = s0 + j;
                if (s < p.C) {
                    const int q = src_slot(s);
                    const uint32_t b = __ldg(vsrc + static_cast<size_t>(q >> 7) * tile + vtile_off(d, q & 127));
                    w[j >> 2] |= b << (8 * (j & 3));
                }
            }
            uint8_t* dst = p.vt_dst + lh * ring + static_cast<size_t>(s0 >> 7) * tile + vtile_off(d, s0 & 127);
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        // scales per (layer, head, slot); write groups per (layer, slot)
        const size_t n = LH * static_cast<size_t>(p.C);
        for (size_t i = i0; i < n; i += stride) {
            const int s = static_cast<int>(i % p.C);
            const size_t lh = i / p.C;
            const size_t o = lh * p.Cpad;
            const int q = src_slot(s);
            p.sk_dst[o + s] = p.sk_src[o + q];
            p.sv_dst[o + s] = p.sv_src[o + q];
            if (lh % p.H == 0) {
                const size_t g = (lh / p.H) * p.Cpad;
                p.grp_dst[g + s] = p.grp_src[g + q];
            }
        }
    }
}

cudaError_t launch_window_shift(const ShiftParams& p, int D, cudaStream_t s) {
    // 8 blocks of 256 threads per SM and part, grid-stride loops over the items
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorUnknown;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cudaErrorUnknown;
    const dim3 grid(8 * sms, 3);
    if (D == 128)
        window_shift_kernel<128><<<grid, 256, 0, s>>>(p);
    else
        window_shift_kernel<64><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace rc
