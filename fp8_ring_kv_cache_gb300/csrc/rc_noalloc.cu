// rc_noalloc.cu -- rc_ring_write_noalloc: the write path (RoPE table kernel +
// fused RoPE/amax/E4M3 write kernel) for callers that cannot allocate device
// memory.  The caller owns the ring buffers and passes them in; the one piece
// of scratch the write needs -- the per-token cos/sin table, plus a copy of
// non-arithmetic positions -- lives in a file-scope __device__ array instead
// of memory from cudaMalloc.  The RoPE frequencies travel in the kernel's
// parameters.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "rc.h"
#include "rc_internal.h"
#include "rc_layout.h"

using namespace rc;

namespace {

constexpr int kNoallocMaxTokens = RC_NOALLOC_MAX_TOKENS;
constexpr int kNoallocMaxHalf = 64;  // head_dim <= 128
constexpr size_t kPosOff = 0;
constexpr size_t kTableOff = kPosOff + sizeof(int64_t) * kNoallocMaxTokens;
constexpr size_t kScratchBytes = kTableOff + sizeof(float2) * kNoallocMaxTokens * kNoallocMaxHalf;
constexpr int kMaxDevices = 64;

}  // namespace

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Device address of g_noalloc_scratch on each device, found once per device
// (by the first call made with that device current).  A cudaDeviceReset of
// the device after that call would leave the address stale; it is not
// supported.
unsigned char* g_scratch_ptr[kMaxDevices] = {};

int scratch_for_current_device(unsigned char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RC_ERR_UNSUPPORTED;
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return RC_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_scratch_ptr[dev];
    return RC_OK;
}

int64_t floormod(int64_t a, int64_t m) {
    int64_t r = a % m;
    return r < 0 ? r + m : r;
}

}  // namespace

extern "C" int rc_ring_write_noalloc(const rc_ring_view* ring, const void* K_bf16, const void* V_bf16,
                                     const int64_t* positions, int n, int64_t delta_total, int32_t group,
                                     double rope_base, void* stream) {
    if (!ring || !K_bf16 || !V_bf16 || !positions) return RC_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(K_bf16) & 15u) || (reinterpret_cast<uintptr_t>(V_bf16) & 15u)) return RC_ERR_ARG;
    if (!ring->kcodes || !ring->vcodes || !ring->kscale || !ring->vscale || !ring->group) return RC_ERR_ARG;
    if (ring->heads < 1 || ring->slots < 1 || !(rope_base > 1.0) || group < 0) return RC_ERR_ARG;
    if (ring->head_dim != 64 && ring->head_dim != 128) return RC_ERR_UNSUPPORTED;
    if (n < 1 || n > ring->slots || n > kNoallocMaxTokens) return RC_ERR_ARG;
    const int C = ring->slots, D = ring->head_dim, half = D / 2;
    // two tokens of one write may not share a slot (slots sorted in a stack array)
    int32_t slots[kNoallocMaxTokens];
    for (int t = 0; t < n; ++t) slots[t] = static_cast<int32_t>(floormod(positions[t] - delta_total, C));
    std::sort(slots, slots + n);
    for (int t = 1; t < n; ++t)
        if (slots[t] == slots[t - 1]) return RC_ERR_ARG;
    unsigned char* scratch = nullptr;
    int st = scratch_for_current_device(&scratch);
    if (st != RC_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    bool arith = true;
    for (int t = 1; t < n; ++t)
        if (positions[t] != positions[0] + t) {
            arith = false;
            break;
        }
    int64_t* dpos = reinterpret_cast<int64_t*>(scratch + kPosOff);
    // pageable host source: the call returns once the positions have been staged
    if (!arith && cudaMemcpyAsync(dpos, positions, sizeof(int64_t) * n, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return RC_ERR_CUDA;
    float2* table = reinterpret_cast<float2*>(scratch + kTableOff);

    RopeTableParams tp{};
    tp.table = table;
    tp.pos = arith ? nullptr : dpos;
    tp.p0 = positions[0];
    for (int i = 0; i < half && i < kNoallocMaxHalf; ++i) tp.theta[i] = std::pow(rope_base, -2.0 * i / D);
    tp.n = n;
    tp.half = half;
    if (launch_rope_table(tp, s) != cudaSuccess) return RC_ERR_CUDA;

    WriteParams wp{};
    wp.kc = ring->kcodes;
    wp.vt = ring->vcodes;
    wp.sk = ring->kscale;
    wp.sv = ring->vscale;
    wp.grp = ring->group;
    wp.K = static_cast<const __nv_bfloat16*>(K_bf16);
    wp.V = static_cast<const __nv_bfloat16*>(V_bf16);
    wp.rope = table;
    wp.pos = arith ? nullptr : dpos;
    wp.p0 = positions[0];
    wp.delta_total = delta_total;
    wp.slot0 = static_cast<int>(floormod(positions[0] - delta_total, C));
    wp.status = nullptr;
    wp.n = n;
    wp.H = ring->heads;
    wp.C = C;
    wp.T = tiles_of(C);
    wp.Cpad = wp.T * kTileSlots;
    wp.group = group;
    if (launch_write(wp, D, s) != cudaSuccess) return RC_ERR_CUDA;
    return RC_OK;
}
