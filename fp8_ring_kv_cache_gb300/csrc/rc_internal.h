// rc_internal.h -- kernel parameter blocks and launchers shared by the host
// layer (rc_host.cu) and the kernel translation units.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace rc {

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device.  The attribute is held per device, so `done` keeps one bit per
// device index (below 64; other devices set it on every launch).
template <typename Kernel>
inline cudaError_t smem_limit_once(Kernel* kernel, uint32_t bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

constexpr int kMaxHalfDim = 64;  // head_dim <= 128

// K1: cos/sin of p * theta_i for the n positions of one write, fp64 angle.
struct RopeTableParams {
    float2* table;         // [n][D/2] (cos, sin)
    const int64_t* pos;    // device positions, or nullptr for p0 + t
    int64_t p0;
    int n;
    int half;              // D/2
    double theta[kMaxHalfDim];  // fp64 frequencies theta_i (by value: no device copy)
};

// K2: fused RoPE + per-head amax + E4M3 quantisation + scatter into ring slots.
struct WriteParams {
    uint8_t* kc;           // layer base [H][T][128][D]
    uint8_t* vt;           // layer base [H][T][D][128]
    float* sk;             // layer base [H][Cpad]
    float* sv;
    int32_t* grp;          // layer base [Cpad]
    const __nv_bfloat16* K;  // [n][H][D]
    const __nv_bfloat16* V;
    const float2* rope;    // [n][D/2]
    const int64_t* pos;    // device positions or nullptr (arithmetic run)
    int64_t p0;
    int64_t delta_total;
    int slot0;             // floormod(p0 - delta_total, C) when pos is nullptr
    int n, H, C, T, Cpad;
    int32_t group;         // compact write-group index of this write
    __nv_bfloat16* kraw;   // read-time store [H][Cpad][D] (nullptr if off)
    __nv_bfloat16* vraw;
    int64_t* slot_pos;     // read-time store: each slot's position [Cpad] (nullptr if off)
    int* status;           // device status word (bounded waits)
};

// K2f: the write fused into the K/V projection: K = k_mul X Wk^T,
// V = v_mul X Wv^T on the tensor cores, then the write of K2 from the fp32
// accumulators.  Uses w's ring, scale, group, RoPE and slot fields (w.K and
// w.V are unused).
constexpr int kFusedMaxTokens = 2048;  // 8 blocks of 256 rows: one portable cluster along M
struct FusedParams {
    WriteParams w;
    float k_mul, v_mul;  // x_scale * wk_scale, x_scale * wv_scale
    int hidden;          // projection input width (a multiple of 64)
    uint64_t wait_ns;    // bound of one device wait
};

// K3: in-place delta rotation with per-(layer, head, group) requantisation.
struct RotateParams {
    uint8_t* kc;           // all layers [L][H][T][128][D]
    float* sk;             // [L][H][Cpad]
    const int32_t* grp;    // [L][Cpad]
    int64_t* slot_pos;     // read-time store [L][Cpad]: moved by delta (nullptr if off)
    int64_t delta;
    int H, C, T, Cpad;
    uint64_t wait_ns;        // bound of one device wait
    float2 cs[kMaxHalfDim];  // (cos, sin) of delta * theta_i
};

// K5: read-time ablation, rebuild one layer's FP8 ring from the bf16 store
// with one scale per head (and per K / V) over every occupied slot.
struct ReadtimeParams {
    const __nv_bfloat16* kraw;  // layer [H][Cpad][D]
    const __nv_bfloat16* vraw;
    const float2* slot_rope;    // [Cpad][D/2]: cos/sin at each slot's current position
    const int32_t* grp;         // layer [Cpad]
    uint8_t* kc;                // scratch ring [H][T][128][D]
    uint8_t* vt;                // [H][T][D][128]
    float* sk;                  // [H][Cpad]
    float* sv;
    int H, C, T, Cpad;
    int* status;                // device status word (index checks of the bounds-checked build)
};

// K4: FP8 attention over one layer's ring (the queries are rotated, scaled
// and split into E4M3 pieces in the kernel's prologue).
struct AttnParams {
    const uint8_t* kc;     // layer [H][T][128][D]
    const uint8_t* vt;     // layer [H][T][D][128]
    const float* sk;       // layer [H][Cpad]
    const float* sv;
    const int32_t* grp;    // layer [Cpad]
    const __nv_bfloat16* q;  // [n][H][D]
    const float2* rope;    // [n][D/2]
    float* out;            // [n][H][D]
    int n, H, C, T, Cpad;
    int masked;            // 1: some slots are empty, read grp
    // bit j: every ring slot of KV tile j (the last tile may hold fewer than
    // 128) is occupied by one write group, so one K and one V scale per head
    // cover the tile; tiles 0..255
    uint64_t uniform[4];
    // tile j (not uniform) made of two write groups, slots [0, b) and [b, 128)
    // of a full tile: split[j] = b (1..127), else 0
    uint8_t split[256];
    float sm_log2;         // log2(e) / sqrt(D)
    int* status;           // device status word
    uint64_t wait_ns;      // limit of one bounded wait (0: give up on any phase not complete)
};

// K6: the copy-based window (an ablation): in every layer, slot s of the
// destination bank takes slot (s + k) mod C of the source bank.
struct ShiftParams {
    const uint8_t* kc_src;     // all layers [L][H][T][128][D]
    uint8_t* kc_dst;
    const uint8_t* vt_src;     // all layers [L][H][T][D][128]
    uint8_t* vt_dst;
    const float* sk_src;       // [L][H][Cpad]
    float* sk_dst;
    const float* sv_src;
    float* sv_dst;
    const int32_t* grp_src;    // [L][Cpad]
    int32_t* grp_dst;
    int L, H, C, T, Cpad;
    int k;                     // 0 < k < C
};

cudaError_t launch_rope_table(const RopeTableParams& p, cudaStream_t s);
cudaError_t launch_window_shift(const ShiftParams& p, int D, cudaStream_t s);
cudaError_t launch_write(const WriteParams& p, int D, cudaStream_t s);
cudaError_t launch_rotate(const RotateParams& p, int D, int layers, cudaStream_t s, int* status);
cudaError_t launch_readtime(const ReadtimeParams& p, int D, cudaStream_t s);
cudaError_t launch_attention(const AttnParams& p, int D, cudaStream_t s);
// the bf16 ring (RC_F_BF16_CACHE): kc / vt hold bf16 tiles, sk / sv are unused
cudaError_t launch_bf16_write(const WriteParams& p, int D, cudaStream_t s);
cudaError_t launch_bf16_rotate(const RotateParams& p, int D, int layers, cudaStream_t s);
cudaError_t launch_bf16_attention(const AttnParams& p, int D, cudaStream_t s);
// the fused projection + write: X [n][hidden], Wk / Wv [H*D][hidden] E4M3 codes
cudaError_t launch_fused_write(const FusedParams& p, const uint8_t* X, const uint8_t* Wk, const uint8_t* Wv, int D,
                               cudaStream_t s);

// Status values a kernel writes into the device status word.
enum DeviceStatus : int {
    kDevOk = 0,
    kDevTimeoutLoader = 101,
    kDevTimeoutMma = 102,
    kDevTimeoutSoftmax = 103,
    kDevTimeoutConvert = 104,
    kDevTimeoutEpilogue = 105,
    kDevBoundsBase = 200,  // + the site of a failed index check (bounds-checked build only)
};

// Sites of the bounds-checked build's index checks (kDevBoundsBase + site).
enum BoundsSite : int {
    kSiteWriteStage = 1,   // K2: a token's K, V rows staged from the inputs
    kSiteWriteRope = 2,    // K2: a token's cos/sin row
    kSiteWriteSlot = 3,    // K2: a token's slot (codes, scales, group, read-time store)
    kSiteWriteVStage = 4,  // K2: the shared-memory V staging row
    kSiteRotCopy = 10,     // K3 staged: the CTA's tiles, scales and groups copied in
    kSiteRotRow = 11,      // K3: a row's codes, scale or position stored back
    kSiteRotGroup = 12,    // K3: a write group's amax table entry
    kSiteAttnTile = 20,    // K4: a K tile with its scales (and groups) copied in
    kSiteAttnQuery = 21,   // K4: a query row read
    kSiteAttnVt = 22,      // K4: a Vt tile read by the converter warps
    kSiteAttnOut = 23,     // K4: an output row stored
    kSiteRtRow = 30,       // K5: a slot's unrotated K, V row and its cos/sin read
    kSiteRtTile = 31,      // K5: a tile's codes and a slot's scales stored
};

}  // namespace rc
