// rc_host.cu -- the C ABI (include/rc.h): handle, ring-slot allocator and index
// math, write-group bookkeeping, RoPE table pool, argument checks, launches,
// and the canonical export used by the tests.
//
// Ring index math (paperdot abstract: "a ring cache"; cpdf.ai "Como rodar 57B
// em tempo real com batch size 1": the window advances without copies): token
// at position p lives in slot floormod(p - delta_total, C).  A delta rotation
// adds delta to every stored position and to delta_total, so no token moves.
#include <algorithm>
#include <utility>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "rc.h"
#include "rc_internal.h"
#include "rc_layout.h"

using namespace rc;

namespace {

constexpr int kPoolEntries = 4;
constexpr int64_t kEmpty = INT64_MIN;

struct RopeEntry {
    bool valid = false;
    bool arith = false;
    int64_t p0 = 0;
    int n = 0;
    std::vector<int64_t> pos;  // the positions (kept for non-arithmetic keys)
    uint64_t stamp = 0;
    float2* d_table = nullptr;  // [max_write][D/2]
    int64_t* d_pos = nullptr;   // [max_write]
    int64_t* h_pos = nullptr;   // pinned staging [max_write]
    cudaEvent_t copied = nullptr;
    bool copy_pending = false;
};

}  // namespace

struct rc_cache {
    rc_config cfg{};
    int device = 0;
    int L = 0, H = 0, D = 0, C = 0, T = 0, Cpad = 0, max_write = 0;
    bool ablation = false;
    bool copy_window = false;  // RC_F_COPY_WINDOW: a second bank for rc_cache_window_shift
    bool bf16 = false;         // RC_F_BF16_CACHE: bf16 tiles in d_kc / d_vt, no scales
    // device memory
    uint8_t* d_kc = nullptr;
    uint8_t* d_vt = nullptr;
    float* d_sk = nullptr;
    float* d_sv = nullptr;
    int32_t* d_grp = nullptr;
    int* d_status = nullptr;
    std::vector<std::pair<void*, size_t>> guarded;  // bounds-checked build: (guarded base, bytes) of each buffer
    __nv_bfloat16* d_kraw = nullptr;
    __nv_bfloat16* d_vraw = nullptr;
    int64_t* d_slot_pos = nullptr;   // [L][Cpad] each slot's current position (read-time store)
    float2* d_rt_rope = nullptr;     // [Cpad][D/2] the read-time call's angle table
    uint8_t* d_rt_kc = nullptr;
    uint8_t* d_rt_vt = nullptr;
    float* d_rt_sk = nullptr;
    float* d_rt_sv = nullptr;
    // the copy-based window's second bank (same shapes as d_kc .. d_grp)
    uint8_t* d2_kc = nullptr;
    uint8_t* d2_vt = nullptr;
    float* d2_sk = nullptr;
    float* d2_sv = nullptr;
    int32_t* d2_grp = nullptr;
    RopeEntry pool[kPoolEntries];
    uint64_t clock = 0;
    // host mirrors of the ring tables
    std::vector<int64_t> pos, gid;        // [L][C]
    std::vector<int32_t> grp;             // [L][C] compact group index, -1 empty
    std::vector<int> occupancy;           // [L]
    std::vector<std::vector<int32_t>> refcnt, freelist;  // per layer
    std::vector<std::vector<int64_t>> last_pos;          // per layer
    std::vector<int> last_n, last_entry;
    std::vector<std::array<uint64_t, 4>> uniform;  // per layer: tiles inside one write group
    std::vector<std::array<uint8_t, 256>> split;   // per layer: two-run tiles (first slot of the second run)
    std::vector<char> uniform_dirty;
    std::vector<uint32_t> slot_mark;
    std::vector<int32_t> wslot;            // [max_write] slots of the write in progress
    uint32_t mark = 0;
    std::vector<double> theta;
    int64_t delta_total = 0, next_gid = 0, launches = 0;
    // sum of the copy-based window's shifts: token at position p lives in
    // slot floormod(p - delta_total - slot_shift, C) (0 for a plain ring)
    int64_t slot_shift = 0;
    cudaStream_t last_stream = nullptr;
    uint64_t wait_ns = 2000000000ull;  // limit of one bounded device wait (rc_cache_set_wait_limit)
};

namespace {

size_t ring_bytes(const rc_cache* h) {
    return static_cast<size_t>(h->L) * h->H * h->T * kTileSlots * h->D * (h->bf16 ? 2 : 1);
}
size_t scale_count(const rc_cache* h) { return h->bf16 ? 0 : static_cast<size_t>(h->L) * h->H * h->Cpad; }

int64_t floormod(int64_t a, int64_t m) {
    int64_t r = a % m;
    return r < 0 ? r + m : r;
}

void dfree(rc_cache* h, void* p);

void free_all(rc_cache* h) {
    if (!h) return;
    cudaSetDevice(h->device);
    dfree(h, h->d_kc);
    dfree(h, h->d_vt);
    dfree(h, h->d_sk);
    dfree(h, h->d_sv);
    dfree(h, h->d_grp);
    dfree(h, h->d_status);
    dfree(h, h->d_kraw);
    dfree(h, h->d_vraw);
    dfree(h, h->d_slot_pos);
    dfree(h, h->d_rt_rope);
    dfree(h, h->d_rt_kc);
    dfree(h, h->d_rt_vt);
    dfree(h, h->d_rt_sk);
    dfree(h, h->d_rt_sv);
    dfree(h, h->d2_kc);
    dfree(h, h->d2_vt);
    dfree(h, h->d2_sk);
    dfree(h, h->d2_sv);
    dfree(h, h->d2_grp);
    for (auto& e : h->pool) {
        dfree(h, e.d_table);
        dfree(h, e.d_pos);
        if (e.h_pos) cudaFreeHost(e.h_pos);
        if (e.copied) cudaEventDestroy(e.copied);
    }
    delete h;
}

// Tiles whose slots are all occupied by a single write group (uniform), and
// full tiles made of two runs, slots [0, b) of one write group and [b, 128) of
// another (split[t] = b, 1..127; 0 for every other tile).  g: the layer's
// group per slot (-1 empty), C slots; tiles past 256 are left unmarked.
void classify_tiles(const int32_t* g, int C, std::array<uint64_t, 4>& m, std::array<uint8_t, 256>& sp) {
    m = {0, 0, 0, 0};
    sp.fill(0);
    const int T = (C + kTileSlots - 1) / kTileSlots;
    for (int t = 0; t < T && t < 256; ++t) {
        // the ring's slots of the tile (the last tile may end before 128)
        const int s0 = t * kTileSlots, s1 = std::min(s0 + kTileSlots, C);
        if (g[s0] < 0) continue;
        int b = s0 + 1;
        while (b < s1 && g[b] == g[s0]) ++b;
        if (b == s1) {
            m[t >> 6] |= 1ull << (t & 63);
            continue;
        }
        if (s1 - s0 != kTileSlots || g[b] < 0) continue;
        int e = b + 1;
        while (e < s1 && g[e] == g[b]) ++e;
        if (e == s1) sp[t] = static_cast<uint8_t>(b - s0);
    }
}

void refresh_uniform(rc_cache* h, int layer) {
    if (!h->uniform_dirty[layer]) return;
    classify_tiles(h->grp.data() + static_cast<size_t>(layer) * h->C, h->C, h->uniform[layer], h->split[layer]);
    h->uniform_dirty[layer] = 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A named NVTX range around each entry point that enqueues work, so that a
// timeline tool (Nsight Systems, or ncu --nvtx --nvtx-include) shows which
// call launched which kernels; with no tool attached the calls do nothing.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Host-side fault injection for the failure-path tests, read from the
// environment at each use: RC_FAULT_INJECT=alloc:K makes the K-th allocation
// (1-based; device or pinned) of an rc_cache_create fail, RC_FAULT_INJECT=launch
// makes every entry point that launches kernels fail with RC_ERR_CUDA after its
// argument checks and before it changes anything.  Unset: nothing is injected.
struct FaultPlan {
    int alloc_at = 0;
    bool launch = false;
};
FaultPlan fault_plan() {
    FaultPlan f;
    const char* e = std::getenv("RC_FAULT_INJECT");
    if (e == nullptr) return f;
    if (std::strncmp(e, "alloc:", 6) == 0) f.alloc_at = std::atoi(e + 6);
    if (std::strcmp(e, "launch") == 0) f.launch = true;
    return f;
}
bool launch_fault() { return fault_plan().launch; }

bool is_arith(const int64_t* p, int n) {
    for (int t = 1; t < n; ++t)
        if (p[t] != p[0] + t) return false;
    return true;
}

// Find or build the RoPE table entry for positions p[0..n).
int rope_entry(rc_cache* h, const int64_t* p, int n, cudaStream_t s, int* err) {
    const bool arith = is_arith(p, n);
    for (int e = 0; e < kPoolEntries; ++e) {
        RopeEntry& r = h->pool[e];
        if (!r.valid || r.n != n || r.arith != arith || r.p0 != p[0]) continue;
        if (!arith && std::memcmp(r.pos.data(), p, sizeof(int64_t) * n) != 0) continue;
        r.stamp = ++h->clock;
        return e;
    }
    int victim = 0;
    for (int e = 1; e < kPoolEntries; ++e)
        if (!h->pool[e].valid || (h->pool[victim].valid && h->pool[e].stamp < h->pool[victim].stamp)) victim = e;
    if (!h->pool[victim].valid) {
        for (int e = 0; e < kPoolEntries; ++e)
            if (!h->pool[e].valid) {
                victim = e;
                break;
            }
    }
    RopeEntry& r = h->pool[victim];
    r.valid = false;
    RopeTableParams tp{};
    tp.table = r.d_table;
    for (int i = 0; i < h->D / 2; ++i) tp.theta[i] = h->theta[i];
    tp.n = n;
    tp.half = h->D / 2;
    if (arith) {
        tp.pos = nullptr;
        tp.p0 = p[0];
        r.pos.clear();
    } else {
        if (r.copy_pending) {
            if (cudaEventSynchronize(r.copied) != cudaSuccess) {
                *err = RC_ERR_CUDA;
                return -1;
            }
            r.copy_pending = false;
        }
        std::memcpy(r.h_pos, p, sizeof(int64_t) * n);
        if (cudaMemcpyAsync(r.d_pos, r.h_pos, sizeof(int64_t) * n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaEventRecord(r.copied, s) != cudaSuccess) {
            *err = RC_ERR_CUDA;
            return -1;
        }
        r.copy_pending = true;
        r.pos.assign(p, p + n);
        tp.pos = r.d_pos;
        tp.p0 = 0;
    }
    if (launch_rope_table(tp, s) != cudaSuccess) {
        *err = RC_ERR_CUDA;
        return -1;
    }
    h->launches += 1;
    r.valid = true;
    r.arith = arith;
    r.p0 = p[0];
    r.n = n;
    r.stamp = ++h->clock;
    return victim;
}

// Device buffers.  The bounds-checked build puts each between two guard zones
// of kGuardBytes filled with kGuardByte (the zone keeps the buffer's 256-byte
// alignment) and records it, so that rc_cache_sync can find writes past either
// end; the normal build allocates the buffer alone.
#ifdef RC_BOUNDS_CHECK
constexpr size_t kGuardBytes = 256;
constexpr unsigned char kGuardByte = 0xA5;
#endif

template <typename T>
int dmalloc(rc_cache* h, T** p, size_t count) {
    if (count == 0) count = 1;
    const size_t bytes = sizeof(T) * count;
#ifdef RC_BOUNDS_CHECK
    unsigned char* base = nullptr;
    if (cudaMalloc(reinterpret_cast<void**>(&base), bytes + 2 * kGuardBytes) != cudaSuccess) return RC_ERR_OOM;
    if (cudaMemset(base, kGuardByte, kGuardBytes) != cudaSuccess ||
        cudaMemset(base + kGuardBytes + bytes, kGuardByte, kGuardBytes) != cudaSuccess) {
        cudaFree(base);
        return RC_ERR_OOM;
    }
    h->guarded.push_back({base, bytes});
    *p = reinterpret_cast<T*>(base + kGuardBytes);
    return RC_OK;
#else
    (void)h;
    return cudaMalloc(reinterpret_cast<void**>(p), bytes) == cudaSuccess ? RC_OK : RC_ERR_OOM;
#endif
}

// Free a buffer from dmalloc (nullptr is ignored).
void dfree(rc_cache* h, void* p) {
    if (p == nullptr) return;
#ifdef RC_BOUNDS_CHECK
    unsigned char* base = static_cast<unsigned char*>(p) - kGuardBytes;
    for (auto& g : h->guarded)
        if (g.first == base) {
            g.first = nullptr;
            cudaFree(base);
            return;
        }
#endif
    (void)h;
    cudaFree(p);
}

// RC_ERR_BOUNDS if a guard zone of any buffer changed (bounds-checked build).
int check_guards(rc_cache* h) {
#ifdef RC_BOUNDS_CHECK
    std::vector<unsigned char> buf(kGuardBytes);
    for (const auto& g : h->guarded) {
        if (g.first == nullptr) continue;
        const unsigned char* base = static_cast<const unsigned char*>(g.first);
        for (const unsigned char* zone : {base, base + kGuardBytes + g.second}) {
            if (cudaMemcpy(buf.data(), zone, kGuardBytes, cudaMemcpyDeviceToHost) != cudaSuccess) return RC_ERR_CUDA;
            for (unsigned char c : buf)
                if (c != kGuardByte) return RC_ERR_BOUNDS;
        }
    }
#else
    (void)h;
#endif
    return RC_OK;
}

int check_sticky() {
    cudaError_t e = cudaPeekAtLastError();
    return e == cudaSuccess ? RC_OK : RC_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* rc_status_string(int status) {
    switch (status) {
        case RC_OK: return "ok";
        case RC_ERR_ARG: return "invalid argument";
        case RC_ERR_STATE: return "call not valid in the cache's current state";
        case RC_ERR_CUDA: return "CUDA error";
        case RC_ERR_OOM: return "out of device memory";
        case RC_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
        case RC_ERR_UNSUPPORTED: return "unsupported shape or device";
        case RC_ERR_BOUNDS: return "an index check or a buffer guard failed (bounds-checked build)";
        default: return "unknown status";
    }
}

int rc_cache_create(const rc_config* cfg, int device, rc_cache** out) {
    if (!out) return RC_ERR_ARG;
    *out = nullptr;
    if (!cfg) return RC_ERR_ARG;
    if (cfg->layers < 1 || cfg->heads < 1 || cfg->slots < 1 || cfg->max_write < 1 || cfg->max_write > cfg->slots ||
        !(cfg->rope_base > 1.0))
        return RC_ERR_ARG;
    if (cfg->head_dim != 64 && cfg->head_dim != 128) return RC_ERR_UNSUPPORTED;
    if (cfg->slots > 32768 || cfg->heads > 65535 || cfg->layers > 65535) return RC_ERR_UNSUPPORTED;
    if ((cfg->flags & RC_F_READTIME_ABLATION) && (cfg->flags & RC_F_COPY_WINDOW)) return RC_ERR_UNSUPPORTED;
    if ((cfg->flags & RC_F_BF16_CACHE) && (cfg->flags & (RC_F_READTIME_ABLATION | RC_F_COPY_WINDOW)))
        return RC_ERR_UNSUPPORTED;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return RC_ERR_ARG;
    cudaDeviceProp prop{};
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return RC_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return RC_ERR_UNSUPPORTED;
    if (cudaSetDevice(device) != cudaSuccess) return RC_ERR_CUDA;

    rc_cache* h = new (std::nothrow) rc_cache();
    if (!h) return RC_ERR_OOM;
    h->cfg = *cfg;
    h->device = device;
    h->L = cfg->layers;
    h->H = cfg->heads;
    h->D = cfg->head_dim;
    h->C = cfg->slots;
    h->T = tiles_of(cfg->slots);
    h->Cpad = h->T * kTileSlots;
    h->max_write = cfg->max_write;
    h->ablation = (cfg->flags & RC_F_READTIME_ABLATION) != 0;
    h->copy_window = (cfg->flags & RC_F_COPY_WINDOW) != 0;
    h->bf16 = (cfg->flags & RC_F_BF16_CACHE) != 0;

    int st = RC_OK;
    const size_t rb = ring_bytes(h), sc = scale_count(h);
    const FaultPlan fault = fault_plan();
    int alloc_no = 0;
    auto injected = [&]() { return fault.alloc_at > 0 && ++alloc_no == fault.alloc_at; };
    auto dmalloc = [&](auto** p, size_t count) { return injected() ? RC_ERR_OOM : ::dmalloc(h, p, count); };
    st |= dmalloc(&h->d_kc, rb);
    st |= dmalloc(&h->d_vt, rb);
    st |= dmalloc(&h->d_sk, sc);
    st |= dmalloc(&h->d_sv, sc);
    st |= dmalloc(&h->d_grp, static_cast<size_t>(h->L) * h->Cpad);
    st |= dmalloc(&h->d_status, 1);
    for (auto& e : h->pool) {
        st |= dmalloc(&e.d_table, static_cast<size_t>(h->max_write) * (h->D / 2));
        st |= dmalloc(&e.d_pos, static_cast<size_t>(h->max_write));
        if (injected() ||
            cudaMallocHost(reinterpret_cast<void**>(&e.h_pos), sizeof(int64_t) * h->max_write) != cudaSuccess)
            st |= RC_ERR_OOM;
        if (cudaEventCreateWithFlags(&e.copied, cudaEventDisableTiming) != cudaSuccess) st |= RC_ERR_OOM;
    }
    if (h->ablation) {
        const size_t raw = static_cast<size_t>(h->L) * h->H * h->Cpad * h->D;
        st |= dmalloc(&h->d_kraw, raw);
        st |= dmalloc(&h->d_vraw, raw);
        st |= dmalloc(&h->d_slot_pos, static_cast<size_t>(h->L) * h->Cpad);
        st |= dmalloc(&h->d_rt_rope, static_cast<size_t>(h->Cpad) * (h->D / 2));
        const size_t one = static_cast<size_t>(h->H) * h->T * kTileSlots * h->D;
        st |= dmalloc(&h->d_rt_kc, one);
        st |= dmalloc(&h->d_rt_vt, one);
        st |= dmalloc(&h->d_rt_sk, static_cast<size_t>(h->H) * h->Cpad);
        st |= dmalloc(&h->d_rt_sv, static_cast<size_t>(h->H) * h->Cpad);
    }
    if (h->copy_window) {
        st |= dmalloc(&h->d2_kc, rb);
        st |= dmalloc(&h->d2_vt, rb);
        st |= dmalloc(&h->d2_sk, sc);
        st |= dmalloc(&h->d2_sv, sc);
        st |= dmalloc(&h->d2_grp, static_cast<size_t>(h->L) * h->Cpad);
    }
    if (st != RC_OK) {
        free_all(h);
        cudaGetLastError();  // clear the allocation error
        return RC_ERR_OOM;
    }
    bool ok = cudaMemset(h->d_kc, 0, rb) == cudaSuccess && cudaMemset(h->d_vt, 0, rb) == cudaSuccess &&
              cudaMemset(h->d_sk, 0, sizeof(float) * sc) == cudaSuccess &&
              cudaMemset(h->d_sv, 0, sizeof(float) * sc) == cudaSuccess &&
              cudaMemset(h->d_grp, 0xFF, sizeof(int32_t) * h->L * h->Cpad) == cudaSuccess &&
              cudaMemset(h->d_status, 0, sizeof(int)) == cudaSuccess;
    if (ok && h->copy_window) {
        ok = cudaMemset(h->d2_kc, 0, rb) == cudaSuccess && cudaMemset(h->d2_vt, 0, rb) == cudaSuccess &&
             cudaMemset(h->d2_sk, 0, sizeof(float) * sc) == cudaSuccess &&
             cudaMemset(h->d2_sv, 0, sizeof(float) * sc) == cudaSuccess &&
             cudaMemset(h->d2_grp, 0xFF, sizeof(int32_t) * h->L * h->Cpad) == cudaSuccess;
    }
    if (ok && h->ablation) {
        const size_t raw = static_cast<size_t>(h->L) * h->H * h->Cpad * h->D;
        ok = cudaMemset(h->d_kraw, 0, raw * 2) == cudaSuccess && cudaMemset(h->d_vraw, 0, raw * 2) == cudaSuccess &&
             cudaMemset(h->d_slot_pos, 0, sizeof(int64_t) * h->L * h->Cpad) == cudaSuccess &&
             cudaMemset(h->d_rt_rope, 0, sizeof(float2) * h->Cpad * (h->D / 2)) == cudaSuccess;
        // the read-time ring's padding slots, like the main ring's, hold zero codes
        const size_t one = static_cast<size_t>(h->H) * h->T * kTileSlots * h->D;
        ok = ok && cudaMemset(h->d_rt_kc, 0, one) == cudaSuccess && cudaMemset(h->d_rt_vt, 0, one) == cudaSuccess &&
             cudaMemset(h->d_rt_sk, 0, sizeof(float) * h->H * h->Cpad) == cudaSuccess &&
             cudaMemset(h->d_rt_sv, 0, sizeof(float) * h->H * h->Cpad) == cudaSuccess;
    }
    h->theta.resize(h->D / 2);
    for (int i = 0; i < h->D / 2; ++i) h->theta[i] = std::pow(cfg->rope_base, -2.0 * i / h->D);
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        free_all(h);
        return RC_ERR_CUDA;
    }
    const size_t lc = static_cast<size_t>(h->L) * h->C;
    h->pos.assign(lc, kEmpty);
    h->gid.assign(lc, kEmpty);
    h->grp.assign(lc, -1);
    h->occupancy.assign(h->L, 0);
    h->refcnt.assign(h->L, std::vector<int32_t>(h->C, 0));
    h->freelist.assign(h->L, std::vector<int32_t>());
    for (int l = 0; l < h->L; ++l) {
        h->freelist[l].reserve(h->C);
        for (int g = h->C - 1; g >= 0; --g) h->freelist[l].push_back(g);
    }
    h->last_pos.assign(h->L, std::vector<int64_t>());
    for (auto& v : h->last_pos) v.reserve(h->max_write);
    h->last_n.assign(h->L, 0);
    h->last_entry.assign(h->L, -1);
    h->uniform.assign(h->L, std::array<uint64_t, 4>{0, 0, 0, 0});
    h->split.assign(h->L, std::array<uint8_t, 256>{});
    h->uniform_dirty.assign(h->L, 1);
    h->slot_mark.assign(h->C, 0);
    h->wslot.assign(h->max_write, 0);
    *out = h;
    return RC_OK;
}

void rc_cache_destroy(rc_cache* h) {
    if (!h) return;
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    free_all(h);
}

// The bookkeeping of a write (slots, RoPE table, write groups) around the
// launch of its kernel: `launch` gets the filled WriteParams (inputs left
// for it to set) and launches on stream s.
extern "C++" {
template <typename Launch>
static int write_common(rc_cache* h, int layer, const int64_t* positions, int n, cudaStream_t s, Launch&& launch) {
    // the tokens' slots: an arithmetic run (the usual write) takes one modulo
    // and its n <= C slots are distinct; any other run is checked slot by slot
    int32_t* sl = h->wslot.data();
    bool arith = true;
    for (int t = 1; t < n && arith; ++t) arith = positions[t] == positions[0] + t;
    if (arith) {
        int32_t s0 = static_cast<int32_t>(floormod(positions[0] - h->delta_total - h->slot_shift, h->C));
        for (int t = 0; t < n; ++t) {
            sl[t] = s0;
            if (++s0 == h->C) s0 = 0;
        }
    } else {
        if (++h->mark == 0) {
            std::fill(h->slot_mark.begin(), h->slot_mark.end(), 0u);
            h->mark = 1;
        }
        for (int t = 0; t < n; ++t) {
            const int64_t slot = floormod(positions[t] - h->delta_total - h->slot_shift, h->C);
            if (h->slot_mark[slot] == h->mark) return RC_ERR_ARG;
            h->slot_mark[slot] = h->mark;
            sl[t] = static_cast<int32_t>(slot);
        }
    }
    if (check_sticky() != RC_OK) return RC_ERR_CUDA;
    if (cudaSetDevice(h->device) != cudaSuccess) return RC_ERR_CUDA;
    int err = RC_OK;
    const int entry = rope_entry(h, positions, n, s, &err);
    if (entry < 0) return err;
    const RopeEntry& re = h->pool[entry];

    // write-group bookkeeping: release the groups whose last slot is overwritten
    const size_t lb = static_cast<size_t>(layer) * h->C;
    auto& rc = h->refcnt[layer];
    auto& fl = h->freelist[layer];
    for (int t = 0; t < n; ++t) {
        const int32_t slot = sl[t];
        const int32_t old = h->grp[lb + slot];
        if (old >= 0) {
            if (--rc[old] == 0) fl.push_back(old);
        } else {
            h->occupancy[layer] += 1;
        }
    }
    const int32_t g = fl.back();
    fl.pop_back();
    rc[g] = n;
    for (int t = 0; t < n; ++t) {
        const int32_t slot = sl[t];
        h->pos[lb + slot] = positions[t];
        h->gid[lb + slot] = h->next_gid;
        h->grp[lb + slot] = g;
    }

    WriteParams wp{};
    const size_t lring = static_cast<size_t>(layer) * h->H * h->T * kTileSlots * h->D * (h->bf16 ? 2 : 1);
    const size_t lsc = static_cast<size_t>(layer) * h->H * h->Cpad;
    wp.kc = h->d_kc + lring;
    wp.vt = h->d_vt + lring;
    wp.sk = h->bf16 ? nullptr : h->d_sk + lsc;
    wp.sv = h->bf16 ? nullptr : h->d_sv + lsc;
    wp.grp = h->d_grp + static_cast<size_t>(layer) * h->Cpad;
    wp.rope = re.d_table;
    wp.pos = re.arith ? nullptr : re.d_pos;
    wp.p0 = positions[0];
    wp.delta_total = h->delta_total + h->slot_shift;  // the kernel's slot mapping
    wp.slot0 = sl[0];
    wp.status = h->d_status;
    wp.n = n;
    wp.H = h->H;
    wp.C = h->C;
    wp.T = h->T;
    wp.Cpad = h->Cpad;
    wp.group = g;
    if (h->ablation) {
        const size_t raw = static_cast<size_t>(layer) * h->H * h->Cpad * h->D;
        wp.kraw = h->d_kraw + raw;
        wp.vraw = h->d_vraw + raw;
        wp.slot_pos = h->d_slot_pos + static_cast<size_t>(layer) * h->Cpad;
    }
    if (launch(wp) != cudaSuccess) return RC_ERR_CUDA;
    h->launches += 1;
    h->last_pos[layer].assign(positions, positions + n);
    h->uniform_dirty[layer] = 1;
    h->last_n[layer] = n;
    h->last_entry[layer] = entry;
    h->next_gid += 1;
    h->last_stream = s;
    return RC_OK;
}

}  // extern "C++"

int rc_cache_write(rc_cache* h, int layer, const void* K_bf16, const void* V_bf16, const int64_t* positions, int n,
                   void* stream) {
    const NvtxRange range("rc_cache_write");
    if (!h || !K_bf16 || !V_bf16 || !positions) return RC_ERR_ARG;
    if (!aligned16(K_bf16) || !aligned16(V_bf16)) return RC_ERR_ARG;
    if (layer < 0 || layer >= h->L || n < 1 || n > h->max_write) return RC_ERR_ARG;
    if (launch_fault()) return RC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return write_common(h, layer, positions, n, s, [&](WriteParams& wp) {
        wp.K = static_cast<const __nv_bfloat16*>(K_bf16);
        wp.V = static_cast<const __nv_bfloat16*>(V_bf16);
        return h->bf16 ? launch_bf16_write(wp, h->D, s) : launch_write(wp, h->D, s);
    });
}

int rc_cache_write_fused(rc_cache* h, int layer, const uint8_t* X, float x_scale, const uint8_t* Wk, float wk_scale,
                         const uint8_t* Wv, float wv_scale, int hidden, const int64_t* positions, int n,
                         void* stream) {
    const NvtxRange range("rc_cache_write_fused");
    if (!h || !X || !Wk || !Wv || !positions) return RC_ERR_ARG;
    if (!aligned16(X) || !aligned16(Wk) || !aligned16(Wv)) return RC_ERR_ARG;
    if (layer < 0 || layer >= h->L || n < 1 || n > h->max_write || n > kFusedMaxTokens) return RC_ERR_ARG;
    if (hidden < 64 || hidden % 64 != 0) return RC_ERR_ARG;
    if (!(x_scale > 0.f) || !(wk_scale > 0.f) || !(wv_scale > 0.f)) return RC_ERR_ARG;
    if (h->bf16 || h->ablation) return RC_ERR_UNSUPPORTED;
    if (launch_fault()) return RC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return write_common(h, layer, positions, n, s, [&](WriteParams& wp) {
        FusedParams fp{};
        fp.w = wp;
        fp.k_mul = x_scale * wk_scale;
        fp.v_mul = x_scale * wv_scale;
        fp.hidden = hidden;
        fp.wait_ns = h->wait_ns;
        return launch_fused_write(fp, X, Wk, Wv, h->D, s);
    });
}

int rc_cache_delta_rotate(rc_cache* h, int64_t delta, void* stream) {
    const NvtxRange range("rc_cache_delta_rotate");
    if (!h) return RC_ERR_ARG;
    if (delta == 0) return RC_OK;
    if (launch_fault()) return RC_ERR_CUDA;
    if (check_sticky() != RC_OK) return RC_ERR_CUDA;
    if (cudaSetDevice(h->device) != cudaSuccess) return RC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    RotateParams rp{};
    rp.kc = h->d_kc;
    rp.sk = h->d_sk;
    rp.grp = h->d_grp;
    rp.slot_pos = h->ablation ? h->d_slot_pos : nullptr;
    rp.delta = delta;
    rp.H = h->H;
    rp.C = h->C;
    rp.T = h->T;
    rp.Cpad = h->Cpad;
    rp.wait_ns = h->wait_ns;
    for (int i = 0; i < h->D / 2; ++i) {
        const double ang = static_cast<double>(delta) * h->theta[i];
        rp.cs[i] = make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
    }
    if ((h->bf16 ? launch_bf16_rotate(rp, h->D, h->L, s) : launch_rotate(rp, h->D, h->L, s, h->d_status)) !=
        cudaSuccess)
        return RC_ERR_CUDA;
    h->launches += 1;
    for (size_t i = 0; i < h->pos.size(); ++i)
        if (h->pos[i] != kEmpty) h->pos[i] += delta;
    for (int l = 0; l < h->L; ++l) {
        for (auto& p : h->last_pos[l]) p += delta;
        h->last_entry[l] = -1;
    }
    h->delta_total += delta;
    h->last_stream = s;
    return RC_OK;
}

int rc_cache_window_shift(rc_cache* h, int64_t k, void* stream) {
    const NvtxRange range("rc_cache_window_shift");
    if (!h || k < 0) return RC_ERR_ARG;
    if (!h->copy_window) return RC_ERR_STATE;
    const int kk = static_cast<int>(k % h->C);
    if (kk == 0) {
        h->slot_shift += k;
        return RC_OK;
    }
    if (launch_fault()) return RC_ERR_CUDA;
    if (check_sticky() != RC_OK) return RC_ERR_CUDA;
    if (cudaSetDevice(h->device) != cudaSuccess) return RC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ShiftParams sp{};
    sp.kc_src = h->d_kc;
    sp.kc_dst = h->d2_kc;
    sp.vt_src = h->d_vt;
    sp.vt_dst = h->d2_vt;
    sp.sk_src = h->d_sk;
    sp.sk_dst = h->d2_sk;
    sp.sv_src = h->d_sv;
    sp.sv_dst = h->d2_sv;
    sp.grp_src = h->d_grp;
    sp.grp_dst = h->d2_grp;
    sp.L = h->L;
    sp.H = h->H;
    sp.C = h->C;
    sp.T = h->T;
    sp.Cpad = h->Cpad;
    sp.k = kk;
    if (launch_window_shift(sp, h->D, s) != cudaSuccess) return RC_ERR_CUDA;
    h->launches += 1;
    std::swap(h->d_kc, h->d2_kc);
    std::swap(h->d_vt, h->d2_vt);
    std::swap(h->d_sk, h->d2_sk);
    std::swap(h->d_sv, h->d2_sv);
    std::swap(h->d_grp, h->d2_grp);
    // the host tables move the same way: slot s takes slot s + kk (mod C)
    for (int l = 0; l < h->L; ++l) {
        const size_t lb = static_cast<size_t>(l) * h->C;
        std::rotate(h->pos.begin() + lb, h->pos.begin() + lb + kk, h->pos.begin() + lb + h->C);
        std::rotate(h->gid.begin() + lb, h->gid.begin() + lb + kk, h->gid.begin() + lb + h->C);
        std::rotate(h->grp.begin() + lb, h->grp.begin() + lb + kk, h->grp.begin() + lb + h->C);
        h->uniform_dirty[l] = 1;
    }
    h->slot_shift += k;
    h->last_stream = s;
    return RC_OK;
}

// The bf16 ring's attention call: every tile whose slots are all occupied takes
// the fast path (no scales, no validity test).
static int attend_bf16(rc_cache* h, int layer, const void* Q_bf16, float* out, int n, void* stream) {
    if (check_sticky() != RC_OK) return RC_ERR_CUDA;
    if (cudaSetDevice(h->device) != cudaSuccess) return RC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int entry = h->last_entry[layer];
    if (entry < 0 || !h->pool[entry].valid || h->pool[entry].n != n || h->pool[entry].p0 != h->last_pos[layer][0] ||
        (!h->pool[entry].arith && h->pool[entry].pos != h->last_pos[layer])) {
        int err = RC_OK;
        entry = rope_entry(h, h->last_pos[layer].data(), n, s, &err);
        if (entry < 0) return err;
        h->last_entry[layer] = entry;
    }
    const size_t lring = static_cast<size_t>(layer) * h->H * h->T * kTileSlots * h->D * 2;
    AttnParams ap{};
    ap.kc = h->d_kc + lring;
    ap.vt = h->d_vt + lring;
    ap.grp = h->d_grp + static_cast<size_t>(layer) * h->Cpad;
    ap.q = static_cast<const __nv_bfloat16*>(Q_bf16);
    ap.rope = h->pool[entry].d_table;
    ap.out = out;
    ap.n = n;
    ap.H = h->H;
    ap.C = h->C;
    ap.T = h->T;
    ap.Cpad = h->Cpad;
    ap.masked = (h->occupancy[layer] < h->C) ? 1 : 0;
    const int32_t* g = h->grp.data() + static_cast<size_t>(layer) * h->C;
    for (int t = 0; t < h->T && t < 256; ++t) {
        const int s0 = t * kTileSlots, s1 = std::min(s0 + kTileSlots, h->C);
        bool occ = true;
        for (int q = s0; q < s1 && occ; ++q) occ = (g[q] >= 0);
        if (occ) ap.uniform[t >> 6] |= 1ull << (t & 63);
    }
    ap.sm_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(h->D)));
    ap.status = h->d_status;
    ap.wait_ns = h->wait_ns;
    if (launch_bf16_attention(ap, h->D, s) != cudaSuccess) return RC_ERR_CUDA;
    h->launches += 1;
    h->last_stream = s;
    return RC_OK;
}

static int attend_common(rc_cache* h, int layer, const void* Q_bf16, float* out, int n, void* stream,
                         bool readtime) {
    const NvtxRange range(readtime ? "rc_attend_readtime" : "rc_attend");
    if (!h || !Q_bf16 || !out) return RC_ERR_ARG;
    if (!aligned16(Q_bf16) || !aligned16(out)) return RC_ERR_ARG;
    if (layer < 0 || layer >= h->L || n < 1) return RC_ERR_ARG;
    if (h->last_n[layer] == 0 || n != h->last_n[layer] || h->occupancy[layer] == 0) return RC_ERR_STATE;
    if (readtime && !h->ablation) return RC_ERR_STATE;
    if (launch_fault()) return RC_ERR_CUDA;
    if (h->bf16) return attend_bf16(h, layer, Q_bf16, out, n, stream);
    if (check_sticky() != RC_OK) return RC_ERR_CUDA;
    if (cudaSetDevice(h->device) != cudaSuccess) return RC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int entry = h->last_entry[layer];
    if (entry < 0 || !h->pool[entry].valid || h->pool[entry].n != n ||
        h->pool[entry].p0 != h->last_pos[layer][0] ||
        (!h->pool[entry].arith && h->pool[entry].pos != h->last_pos[layer])) {
        int err = RC_OK;
        entry = rope_entry(h, h->last_pos[layer].data(), n, s, &err);
        if (entry < 0) return err;
        h->last_entry[layer] = entry;
    } else {
        h->pool[entry].stamp = ++h->clock;
    }
    const size_t lring = static_cast<size_t>(layer) * h->H * h->T * kTileSlots * h->D;
    const size_t lsc = static_cast<size_t>(layer) * h->H * h->Cpad;
    AttnParams ap{};
    if (readtime) {
        // RoPE at every slot's current position: the angle table of this call
        // (fp64 angles, as for a write) from the device copy of the positions
        RopeTableParams tp{};
        tp.table = h->d_rt_rope;
        tp.pos = h->d_slot_pos + static_cast<size_t>(layer) * h->Cpad;
        tp.p0 = 0;
        for (int i = 0; i < h->D / 2; ++i) tp.theta[i] = h->theta[i];
        tp.n = h->C;
        tp.half = h->D / 2;
        if (launch_rope_table(tp, s) != cudaSuccess) return RC_ERR_CUDA;
        h->launches += 1;
        ReadtimeParams rp{};
        const size_t raw = static_cast<size_t>(layer) * h->H * h->Cpad * h->D;
        rp.kraw = h->d_kraw + raw;
        rp.vraw = h->d_vraw + raw;
        rp.slot_rope = h->d_rt_rope;
        rp.grp = h->d_grp + static_cast<size_t>(layer) * h->Cpad;
        rp.kc = h->d_rt_kc;
        rp.vt = h->d_rt_vt;
        rp.sk = h->d_rt_sk;
        rp.sv = h->d_rt_sv;
        rp.H = h->H;
        rp.C = h->C;
        rp.T = h->T;
        rp.Cpad = h->Cpad;
        rp.status = h->d_status;
        if (launch_readtime(rp, h->D, s) != cudaSuccess) return RC_ERR_CUDA;
        h->launches += 1;
        ap.kc = h->d_rt_kc;
        ap.vt = h->d_rt_vt;
        ap.sk = h->d_rt_sk;
        ap.sv = h->d_rt_sv;
    } else {
        ap.kc = h->d_kc + lring;
        ap.vt = h->d_vt + lring;
        ap.sk = h->d_sk + lsc;
        ap.sv = h->d_sv + lsc;
    }
    ap.grp = h->d_grp + static_cast<size_t>(layer) * h->Cpad;
    ap.q = static_cast<const __nv_bfloat16*>(Q_bf16);
    ap.rope = h->pool[entry].d_table;
    ap.out = out;
    ap.n = n;
    ap.H = h->H;
    ap.C = h->C;
    ap.T = h->T;
    ap.Cpad = h->Cpad;
    ap.masked = (h->occupancy[layer] < h->C) ? 1 : 0;
    if (readtime) {
        // the read-time ring has one scale per head: every fully occupied tile qualifies
        for (int w = 0; w < 4; ++w) ap.uniform[w] = 0;
        const int32_t* g = h->grp.data() + static_cast<size_t>(layer) * h->C;
        for (int t = 0; t < h->T && t < 256; ++t) {
            const int s0 = t * kTileSlots, s1 = std::min(s0 + kTileSlots, h->C);
            bool occ = true;
            for (int s = s0; s < s1 && occ; ++s) occ = (g[s] >= 0);
            if (occ) ap.uniform[t >> 6] |= 1ull << (t & 63);
        }
        std::memset(ap.split, 0, sizeof(ap.split));
    } else {
        refresh_uniform(h, layer);
        for (int w = 0; w < 4; ++w) ap.uniform[w] = h->uniform[layer][w];
        std::memcpy(ap.split, h->split[layer].data(), sizeof(ap.split));
    }
    ap.sm_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(h->D)));
    ap.status = h->d_status;
    ap.wait_ns = h->wait_ns;
    if (launch_attention(ap, h->D, s) != cudaSuccess) return RC_ERR_CUDA;
    h->launches += 1;
    h->last_stream = s;
    return RC_OK;
}

int rc_attend(rc_cache* h, int layer, const void* Q_bf16, float* out_f32, int n, void* stream) {
    return attend_common(h, layer, Q_bf16, out_f32, n, stream, false);
}

int rc_attend_readtime(rc_cache* h, int layer, const void* Q_bf16, float* out_f32, int n, void* stream) {
    return attend_common(h, layer, Q_bf16, out_f32, n, stream, true);
}

int rc_cache_sync(rc_cache* h) {
    if (!h) return RC_ERR_ARG;
    if (cudaSetDevice(h->device) != cudaSuccess) return RC_ERR_CUDA;
    if (cudaStreamSynchronize(h->last_stream) != cudaSuccess) return RC_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return RC_ERR_CUDA;
    int st = 0;
    if (cudaMemcpy(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return RC_ERR_CUDA;
    if (st != 0) {
        cudaMemset(h->d_status, 0, sizeof(int));
        return (st >= rc::kDevBoundsBase && st < rc::kDevBoundsBase + 100) ? RC_ERR_BOUNDS : RC_ERR_TIMEOUT;
    }
    return check_guards(h);
}

unsigned rc_build_flags(void) {
#ifdef RC_BOUNDS_CHECK
    return RC_BUILD_BOUNDS_CHECK;
#else
    return 0u;
#endif
}

static int export_ring(rc_cache* h, const uint8_t* d_kc, const uint8_t* d_vt, const float* d_sk, const float* d_sv,
                       uint8_t* kcodes, float* kscale, uint8_t* vcodes, float* vscale) {
    const int H = h->H, D = h->D, C = h->C, T = h->T, Cp = h->Cpad;
    const size_t one = static_cast<size_t>(H) * T * kTileSlots * D;
    std::vector<uint8_t> buf;
    if (kcodes) {
        buf.resize(one);
        if (cudaMemcpy(buf.data(), d_kc, one, cudaMemcpyDeviceToHost) != cudaSuccess) return RC_ERR_CUDA;
        for (int hh = 0; hh < H; ++hh)
            for (int s = 0; s < C; ++s) {
                const uint8_t* tile = buf.data() + (static_cast<size_t>(hh) * T + s / kTileSlots) * kTileSlots * D;
                uint8_t* dst = kcodes + (static_cast<size_t>(hh) * C + s) * D;
                for (int d = 0; d < D; ++d) dst[d] = tile[ktile_off(s % kTileSlots, d, D)];
            }
    }
    if (vcodes) {
        buf.resize(one);
        if (cudaMemcpy(buf.data(), d_vt, one, cudaMemcpyDeviceToHost) != cudaSuccess) return RC_ERR_CUDA;
        for (int hh = 0; hh < H; ++hh)
            for (int s = 0; s < C; ++s) {
                const uint8_t* tile = buf.data() + (static_cast<size_t>(hh) * T + s / kTileSlots) * kTileSlots * D;
                uint8_t* dst = vcodes + (static_cast<size_t>(hh) * C + s) * D;
                for (int d = 0; d < D; ++d) dst[d] = tile[vtile_off(d, s % kTileSlots)];
            }
    }
    std::vector<float> sbuf;
    if (kscale || vscale) sbuf.resize(static_cast<size_t>(H) * Cp);
    if (kscale) {
        if (cudaMemcpy(sbuf.data(), d_sk, sizeof(float) * sbuf.size(), cudaMemcpyDeviceToHost) != cudaSuccess)
            return RC_ERR_CUDA;
        for (int hh = 0; hh < H; ++hh)
            std::memcpy(kscale + static_cast<size_t>(hh) * C, sbuf.data() + static_cast<size_t>(hh) * Cp,
                        sizeof(float) * C);
    }
    if (vscale) {
        if (cudaMemcpy(sbuf.data(), d_sv, sizeof(float) * sbuf.size(), cudaMemcpyDeviceToHost) != cudaSuccess)
            return RC_ERR_CUDA;
        for (int hh = 0; hh < H; ++hh)
            std::memcpy(vscale + static_cast<size_t>(hh) * C, sbuf.data() + static_cast<size_t>(hh) * Cp,
                        sizeof(float) * C);
    }
    return RC_OK;
}

// The stored fp16 value as bf16 bits, rounded to nearest even (exact for every
// value that came from a bf16 input inside fp16's range).
static uint16_t f16_to_bf16_bits(uint16_t h) {
    const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
    const uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
    uint32_t f;
    if (e == 0x1Fu) {
        f = sign | 0x7F800000u | (m << 13);
    } else if (e != 0) {
        f = sign | ((e + 112u) << 23) | (m << 13);
    } else if (m == 0) {
        f = sign;
    } else {  // subnormal: m * 2^-24
        int sh = 0;
        uint32_t mm = m;
        while ((mm & 0x400u) == 0) {
            mm <<= 1;
            ++sh;
        }
        f = sign | (static_cast<uint32_t>(113 - sh) << 23) | ((mm & 0x3FFu) << 13);
    }
    const uint32_t lsb = (f >> 16) & 1u;
    if ((f & 0x7F800000u) == 0x7F800000u) return static_cast<uint16_t>(f >> 16);
    return static_cast<uint16_t>((f + 0x7FFFu + lsb) >> 16);
}

int rc_cache_export_bf16(rc_cache* h, int layer, uint16_t* kbits, uint16_t* vbits, int64_t* pos, int64_t* gid) {
    if (!h || layer < 0 || layer >= h->L) return RC_ERR_ARG;
    if (!h->bf16) return RC_ERR_STATE;
    int st = rc_cache_sync(h);
    if (st != RC_OK) return st;
    const int H = h->H, D = h->D, C = h->C, T = h->T;
    const size_t tile = static_cast<size_t>(kTileSlots) * D * 2;
    const size_t one = static_cast<size_t>(H) * T * tile;
    const size_t lring = static_cast<size_t>(layer) * one;
    std::vector<uint8_t> buf(one);
    if (kbits) {
        if (cudaMemcpy(buf.data(), h->d_kc + lring, one, cudaMemcpyDeviceToHost) != cudaSuccess) return RC_ERR_CUDA;
        for (int hh = 0; hh < H; ++hh)
            for (int sl = 0; sl < C; ++sl) {
                const uint8_t* t = buf.data() + (static_cast<size_t>(hh) * T + sl / kTileSlots) * tile;
                for (int d = 0; d < D; ++d)
                    std::memcpy(kbits + (static_cast<size_t>(hh) * C + sl) * D + d, t + bktile_off(sl % kTileSlots, d), 2);
            }
    }
    if (vbits) {
        if (cudaMemcpy(buf.data(), h->d_vt + lring, one, cudaMemcpyDeviceToHost) != cudaSuccess) return RC_ERR_CUDA;
        for (int hh = 0; hh < H; ++hh)
            for (int sl = 0; sl < C; ++sl) {
                const uint8_t* t = buf.data() + (static_cast<size_t>(hh) * T + sl / kTileSlots) * tile;
                for (int d = 0; d < D; ++d) {
                    uint16_t f16;
                    std::memcpy(&f16, t + bvtile_off(d, sl % kTileSlots, D), 2);
                    vbits[(static_cast<size_t>(hh) * C + sl) * D + d] = f16_to_bf16_bits(f16);
                }
            }
    }
    const size_t lb = static_cast<size_t>(layer) * h->C;
    if (pos) std::memcpy(pos, h->pos.data() + lb, sizeof(int64_t) * h->C);
    if (gid) std::memcpy(gid, h->gid.data() + lb, sizeof(int64_t) * h->C);
    return RC_OK;
}

int rc_cache_export(rc_cache* h, int layer, uint8_t* kcodes, float* kscale, uint8_t* vcodes, float* vscale,
                    int64_t* pos, int64_t* gid) {
    if (!h || layer < 0 || layer >= h->L) return RC_ERR_ARG;
    if (h->bf16) return RC_ERR_STATE;
    int st = rc_cache_sync(h);
    if (st != RC_OK) return st;
    const size_t lring = static_cast<size_t>(layer) * h->H * h->T * kTileSlots * h->D;
    const size_t lsc = static_cast<size_t>(layer) * h->H * h->Cpad;
    st = export_ring(h, h->d_kc + lring, h->d_vt + lring, h->d_sk + lsc, h->d_sv + lsc, kcodes, kscale, vcodes,
                     vscale);
    if (st != RC_OK) return st;
    const size_t lb = static_cast<size_t>(layer) * h->C;
    if (pos) std::memcpy(pos, h->pos.data() + lb, sizeof(int64_t) * h->C);
    if (gid) std::memcpy(gid, h->gid.data() + lb, sizeof(int64_t) * h->C);
    return RC_OK;
}

int rc_cache_export_readtime(rc_cache* h, uint8_t* kcodes, float* kscale, uint8_t* vcodes, float* vscale) {
    if (!h) return RC_ERR_ARG;
    if (!h->ablation) return RC_ERR_STATE;
    int st = rc_cache_sync(h);
    if (st != RC_OK) return st;
    return export_ring(h, h->d_rt_kc, h->d_rt_vt, h->d_rt_sk, h->d_rt_sv, kcodes, kscale, vcodes, vscale);
}

int rc_cache_occupancy(const rc_cache* h, int layer) {
    if (!h || layer < 0 || layer >= h->L) return RC_ERR_ARG;
    return h->occupancy[layer];
}

int64_t rc_cache_delta_total(const rc_cache* h) { return h ? h->delta_total : 0; }

int rc_cache_set_wait_limit(rc_cache* h, uint64_t ns) {
    if (!h || ns > 60000000000ull) return RC_ERR_ARG;
    h->wait_ns = ns;
    return RC_OK;
}

int64_t rc_cache_launch_count(const rc_cache* h) { return h ? h->launches : 0; }

int rc_tile_kinds(const int32_t* grp, int slots, uint64_t* uniform, uint8_t* split) {
    if (!grp || !uniform || !split || slots < 1 || slots > 32768) return RC_ERR_ARG;
    std::array<uint64_t, 4> m;
    std::array<uint8_t, 256> sp;
    classify_tiles(grp, slots, m, sp);
    std::memcpy(uniform, m.data(), sizeof(m));
    std::memcpy(split, sp.data(), sizeof(sp));
    return RC_OK;
}

}  // extern "C"
