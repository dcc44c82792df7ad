/*
 * rc.h -- C ABI of the write-time FP8 ring KV cache for one GB300 (sm_103a).
 *
 * The operations come from the pages about "Runway Characters: Serving a 57B
 * Video Diffusion Transformer for Real-Time Conversation" (arXiv 2611.05642):
 *   - paperdot abstract mirror: the cache is a ring; keys get RoPE and FP8
 *     quantisation a single time, when written; a reset of the positions
 *     rotates the stored keys by the difference.  A chunk's 240 attention
 *     calls each read 5,788 slots, 757 of them new.
 *   - cpdf.ai blog, section "Como rodar 57B em tempo real com batch size 1":
 *     rotary positions and FP8 quantisation move from read time to write
 *     time, and the ring advances the window without copies.
 *   - cpdf.ai blog, section "Blackwell, escalabilidade e limites do
 *     decodificador": the FP8 attention kernel uses per-head scales.
 *
 * Conventions shared by every call:
 *   - Status: 0 (RC_OK) or a negative RC_ERR_* code.  Argument and state
 *     errors are found on the host before anything is launched, and leave the
 *     cache unchanged.  Errors of kernels already launched surface as
 *     RC_ERR_CUDA from a later call, or from rc_cache_sync.  No C++ exception
 *     crosses this boundary.
 *   - Device pointers are plain CUDA device addresses (for example a torch
 *     tensor's data_ptr()), 16-byte aligned (RC_ERR_ARG otherwise).  The
 *     caller keeps them alive until the work on `stream` that reads or
 *     writes them has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls on one handle must be issued on one stream, or ordered
 *     by the caller; a handle is not thread-safe.
 *   - Memory: rc_cache_create allocates every device and pinned host buffer
 *     the handle will ever use.  No later call allocates, for any write size
 *     up to max_write.
 *   - Layouts: K, V and Q are bf16, token-major [n][heads][head_dim] with
 *     head_dim contiguous.  The attention output is fp32 with the same layout.
 *     head_dim is 64 or 128.
 *   - CUDA graphs: rc_cache_write, rc_attend and rc_cache_delta_rotate only
 *     launch kernels on `stream` once each has been called directly on the
 *     device (the first call sets kernel attributes), so a run of them can be
 *     captured into a graph.  A write to capture must have consecutive
 *     positions (p0, p0 + 1, ...) or repeat the positions of a recent write:
 *     any other position vector goes to the device through a pinned buffer
 *     guarded by an event, which a capture cannot hold.  The host-side
 *     bookkeeping (slots, write groups, the positions the next attention
 *     rotates its queries at) is done when a call is captured, and the graph
 *     keeps that call's arguments: launch each captured graph once, in the
 *     order of capture, with no direct call on the handle in between.
 */
#ifndef RC_H
#define RC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define RC_OK 0
#define RC_ERR_ARG (-1)         /* bad argument: null pointer, size or index out of range,
                                   two tokens of one write on the same slot */
#define RC_ERR_STATE (-2)       /* call not valid in the current state: attention on a
                                   layer never written, or query count different from
                                   that layer's last write */
#define RC_ERR_CUDA (-3)        /* a CUDA runtime call or a launched kernel failed */
#define RC_ERR_OOM (-4)         /* rc_cache_create could not allocate */
#define RC_ERR_TIMEOUT (-5)     /* a kernel gave up a bounded wait and returned early;
                                   its output is not valid */
#define RC_ERR_UNSUPPORTED (-6) /* shape not supported (head_dim other than 64 or 128,
                                   or a device that is not sm_103) */
#define RC_ERR_BOUNDS (-7)      /* bounds-checked build only (rc_build_flags): a kernel's
                                   index check failed and the access was skipped, or a
                                   buffer's guard bytes were overwritten; results are
                                   not valid */

/* ---- configuration ------------------------------------------------------ */
/* Keep the unrotated bf16 K, V of every slot as well, so that rc_attend_readtime
   can redo RoPE and quantisation of the whole cache at read time. */
#define RC_F_READTIME_ABLATION 1u
/* Allocate a second bank of rings so that rc_cache_window_shift can move the
   stored tokens the way a concatenating cache would (the copy-based window
   ablation; doubles the ring memory; not combinable with the flag above). */
#define RC_F_COPY_WINDOW 2u
/* A 16-bit ring instead of E4M3 + per-slot scales: the non-FP8 cache of the
   comparison in the cpdf.ai blog, section "Blackwell, escalabilidade e
   limites do decodificador" (FP8 saves time on H100 and costs time on B200
   without an FP8 attention kernel).  Writes round RoPE(K) once to bf16 and
   store V converted once to fp16 (exact for 2^-17 <= |v| < 65520 and zero;
   smaller magnitudes round to fp16's subnormal step, larger ones become
   +-inf); delta rotations re-rotate every stored key and round it back to
   bf16; attention computes softmax(Q K^T / sqrt(d)) V with fp32 accumulation.
   Doubles the ring memory, keeps no scales; rc_cache_export_bf16 replaces
   rc_cache_export.  Not combinable with the two flags above. */
#define RC_F_BF16_CACHE 4u

typedef struct rc_config {
    int layers;       /* attention layers with one ring each (>= 1) */
    int heads;        /* heads per layer (>= 1) */
    int head_dim;     /* 64 or 128 */
    int slots;        /* ring capacity C per layer (>= 1) */
    int max_write;    /* largest n of one write (1 .. slots) */
    double rope_base; /* RoPE base; theta_i = base^(-2i/head_dim) (> 1) */
    unsigned flags;   /* RC_F_* */
} rc_config;

typedef struct rc_cache rc_cache; /* opaque; owns all of its memory */

/*
 * Create a cache on CUDA device `device` and store the handle in *out.
 * Every slot starts empty.  Allocates the FP8 rings (2 * layers * heads *
 * ceil(slots/128)*128 * head_dim bytes), the per-slot scales, the RoPE table
 * pool and the pinned position staging, and with RC_F_READTIME_ABLATION the
 * bf16 store.  On error *out is NULL and nothing is leaked.
 */
int rc_cache_create(const rc_config *cfg, int device, rc_cache **out);

/*
 * Write n new tokens into ring `layer` (paperdot abstract: RoPE and FP8
 * quantisation happen here, a single time per token).  K_bf16 and V_bf16 are device
 * pointers to [n][heads][head_dim] bf16.  positions is a HOST array of n
 * int64 token positions (any sign).  Token t goes to slot
 * floormod(positions[t] - delta_total, slots), replacing what was there.
 * For every head, K is rotated by RoPE at its position; then K and V each get
 * one fp32 scale s = fl32(amax/448) over the n tokens of that head (s = 1 if
 * amax = 0), and each element is stored as the E4M3 code of fl32(x/s),
 * rounded to nearest even and saturated to +-448.
 * Errors: RC_ERR_ARG if layer is out of range, n < 1 or n > max_write, a
 * pointer is NULL, or two tokens map to one slot.
 * A position vector that is not an arithmetic run p0, p0+1, ... is copied to
 * the device through pinned staging; an arithmetic run needs no copy.
 */
int rc_cache_write(rc_cache *h, int layer, const void *K_bf16, const void *V_bf16,
                   const int64_t *positions, int n, void *stream);

/*
 * Position reset (paperdot abstract: resetting the positions rotates the
 * stored keys by the difference).  Every occupied slot of every layer moves from position p to
 * p + delta without moving slots: the stored keys are dequantised, rotated
 * by delta, and each (layer, head, write group) is requantised in place with
 * a fresh scale from its new amax.  Values are untouched.  The layers' last
 * write positions move by delta too.  delta = 0 is a no-op.
 */
int rc_cache_delta_rotate(rc_cache *h, int64_t delta, void *stream);

/*
 * The copy-based window, an ablation of the ring (paperdot abstract: the
 * window advances "without copies"; this is the copy).  A cache that keeps
 * its tokens in position order moves them k slots down when k new positions
 * arrive, then writes the new tokens at the end.  This call does that move in
 * every layer: slot s takes what slot (s + k) mod slots held (K and V codes,
 * their scales and write groups, one read and one write of every ring, into
 * the second bank), and from then on a token at position p lives in slot
 * floormod(p - delta_total - (sum of shifts), slots).  The set of stored
 * tokens, their codes and every attention result are those of the ring;
 * rc_cache_export returns the slots in their shifted order.  k = 0 (or a
 * multiple of slots) moves nothing.
 * Errors: RC_ERR_STATE unless the cache was created with RC_F_COPY_WINDOW;
 * RC_ERR_ARG for a NULL handle or k < 0.
 */
int rc_cache_window_shift(rc_cache *h, int64_t k, void *stream);

/*
 * Attention call (paperdot abstract: the new tokens' queries read the whole
 * cache).  Q_bf16 is a device pointer to [n][heads][head_dim] bf16 queries of
 * the layer's last write; each is rotated at that token's (current) position.
 * out_f32 is a device pointer to [n][heads][head_dim] fp32:
 *   out = softmax(q . k_j / sqrt(head_dim)) over the occupied slots j, times v_j,
 * with k_j, v_j the stored codes times their slot's scale.  No mask.
 * Errors: RC_ERR_STATE if the layer was never written or n differs from the
 * layer's last write; RC_ERR_ARG for NULL pointers or a bad layer.
 */
int rc_attend(rc_cache *h, int layer, const void *Q_bf16, float *out_f32, int n,
              void *stream);

/*
 * Read-time ablation of rc_attend (the original design the pages describe
 * in the abstract and in the cpdf.ai section "Como rodar 57B em tempo real
 * com batch size 1": RoPE and FP8 quantisation of the WHOLE cache redone in
 * every attention call).  Rebuilds this layer's FP8 ring from the unrotated
 * bf16 store into a scratch ring, then runs the same attention kernel on it.
 * Every stored key is rotated at its slot's CURRENT position: the store keeps
 * each slot's position on the device and rc_cache_delta_rotate moves it, so
 * after any number of resets the read-time ring holds the keys the write-time
 * ring would hold had it been written at today's positions.  Each call first
 * rebuilds the angle table of all slots (fp64 angles) from those positions.
 * Requires RC_F_READTIME_ABLATION, else RC_ERR_STATE.  The read-time ring
 * quantises each head with ONE scale over all occupied slots (per K and V),
 * so its codes differ from the write-time ring's wherever that ring holds
 * several write groups with different scales; the rotated keys before
 * quantisation are the same.
 */
int rc_attend_readtime(rc_cache *h, int layer, const void *Q_bf16, float *out_f32,
                       int n, void *stream);

/* Free everything the handle owns (waits for its device work first). NULL is ignored. */
void rc_cache_destroy(rc_cache *h);

/* A static description of a status code. */
const char *rc_status_string(int status);

/* ---- inspection and test support -------------------------------------- */

/* Synchronise the handle's last stream and report any kernel error or timeout
   (RC_ERR_TIMEOUT), and in the bounds-checked build a failed index check or
   overwritten guard bytes (RC_ERR_BOUNDS).  The device status word is cleared. */
int rc_cache_sync(rc_cache *h);

/* How this library was built: RC_BUILD_BOUNDS_CHECK is set in the bounds-
   checked build (librc_bounds.so, compiled with -DRC_BOUNDS_CHECK).  There,
   the write, rotation, read-time and attention kernels test the index of each global
   access they make against the buffer it addresses before making it (a
   failure skips the access and records the site; nothing traps), and every
   device buffer of a handle sits between two 256-byte guard zones filled with
   0xA5 that rc_cache_sync checks.  The normal build has neither and returns 0.
   Needs no device. */
#define RC_BUILD_BOUNDS_CHECK 1u
unsigned rc_build_flags(void);

/*
 * Failure-path support.  Every wait inside the attention kernel is bounded:
 * past `ns` nanoseconds (default 2 s) the kernel gives up, records where, frees
 * its tensor memory and returns, and the next rc_cache_sync reports
 * RC_ERR_TIMEOUT (and clears the record; the ring itself is not modified by an
 * attention call, so the handle stays usable).  ns = 0 gives up on any wait
 * whose phase is not already complete, which makes a wait run out on purpose.
 * Errors: RC_ERR_ARG for a NULL handle or ns above 60 s.
 *
 * Host-side fault injection, read from the environment at each use:
 * RC_FAULT_INJECT=alloc:K makes the K-th allocation (1-based, device or
 * pinned) of rc_cache_create fail, which then returns RC_ERR_OOM having freed
 * everything it had allocated; RC_FAULT_INJECT=launch makes every call that
 * launches kernels return RC_ERR_CUDA after its argument checks, before it
 * changes anything.
 */
int rc_cache_set_wait_limit(rc_cache *h, uint64_t ns);

/*
 * Write n new tokens into ring `layer` straight from the K/V projection: the
 * write fused into the projection's FP8 GEMM (the single-GPU half of the
 * pages' fused FP8 GEMM: paperdot abstract; cpdf.ai blog, "Como rodar 57B em
 * tempo real com batch size 1").  With X, Wk, Wv E4M3 codes and one scale
 * each,
 *   K[t][h][i] = x_scale * wk_scale * sum_k X[t][k] * Wk[h*head_dim + i][k]
 * and V likewise with Wv, wv_scale, computed on the tensor cores (fp32
 * accumulation); then written as rc_cache_write writes its K and V (RoPE at
 * positions[t], one scale per head for K and for V, E4M3 codes into the
 * slots), from the fp32 products with no bf16 rounding in between.
 * X: device [n][hidden] uint8, row stride hidden bytes; Wk, Wv: device
 * [heads*head_dim][hidden] uint8 (one weight row per output feature); all
 * 16-byte aligned.  hidden: a multiple of 64.  positions: HOST int64 [n], as
 * for rc_cache_write.  Stream-ordered; the caller keeps X, Wk, Wv alive until
 * the work on `stream` has finished.
 * A fused write whose kernel gave up a bounded wait (rc_cache_sync then reports
 * RC_ERR_TIMEOUT) leaves its slots undefined; writing them again repairs them.
 * Errors: RC_ERR_ARG (a pointer NULL or unaligned, layer out of range, n < 1,
 * n > max_write or n > 2048, hidden not a positive multiple of 64, a scale not
 * positive, two tokens on one slot); RC_ERR_UNSUPPORTED with RC_F_BF16_CACHE
 * or RC_F_READTIME_ABLATION (the read-time store keeps bf16 K and V, which
 * this path never forms).
 */
int rc_cache_write_fused(rc_cache *h, int layer, const uint8_t *X, float x_scale,
                         const uint8_t *Wk, float wk_scale, const uint8_t *Wv, float wv_scale,
                         int hidden, const int64_t *positions, int n, void *stream);

/*
 * Copy ring `layer` to HOST buffers in canonical layout (synchronous):
 * kcodes, vcodes: uint8 [heads][slots][head_dim] E4M3 codes; kscale, vscale:
 * fp32 [heads][slots]; pos: int64 [slots] position (INT64_MIN = empty);
 * gid: int64 [slots] serial number of the write that filled the slot
 * (INT64_MIN = empty; writes are numbered 0, 1, ... per handle).  Any
 * pointer may be NULL to skip that table.
 */
int rc_cache_export(rc_cache *h, int layer, uint8_t *kcodes, float *kscale,
                    uint8_t *vcodes, float *vscale, int64_t *pos, int64_t *gid);

/*
 * Copy the scratch ring that the last rc_attend_readtime call built (same
 * canonical layouts as rc_cache_export; synchronous).  RC_ERR_STATE without
 * RC_F_READTIME_ABLATION.
 */
int rc_cache_export_readtime(rc_cache *h, uint8_t *kcodes, float *kscale,
                             uint8_t *vcodes, float *vscale);

/*
 * Copy ring `layer` of a RC_F_BF16_CACHE cache to HOST buffers (synchronous):
 * kbits, vbits: uint16 [heads][slots][head_dim] bf16 bit patterns (RoPE'd keys
 * at their current positions; the stored fp16 values rounded to bf16, which
 * returns each in-range value as written; zeros in empty slots); pos,
 * gid as in rc_cache_export.  Any pointer may be NULL.  RC_ERR_STATE without
 * the flag (and rc_cache_export answers RC_ERR_STATE with it).
 */
int rc_cache_export_bf16(rc_cache *h, int layer, uint16_t *kbits, uint16_t *vbits,
                         int64_t *pos, int64_t *gid);

/* ---- allocation-free write into a caller-owned ring -------------------- */
/*
 * No counterpart in the paper: this is an integration convenience.
 *
 * Some callers cannot call cudaMalloc: a process whose device memory is all
 * reserved up front by another allocator (a framework's caching allocator or
 * a fixed arena), where a new allocation would fail or fragment that pool; or
 * a latency-critical loop that must never pay for cudaMalloc / cudaFree, which
 * can synchronise the whole device.  rc_ring_write_noalloc serves them: it
 * performs exactly the write of rc_cache_write (RoPE table kernel, then the
 * fused RoPE + per-head amax + E4M3 write kernel) into ring buffers that the
 * CALLER owns, and it allocates nothing.  Its only scratch -- a copy of
 * non-arithmetic positions and the per-token cos/sin table -- lives in one
 * file-scope __device__ array of about 2 MiB (RC_NOALLOC_MAX_TOKENS tokens x
 * 64 pairs x 8 bytes, plus 32 KiB), which every GPU that loads the library
 * holds until the process exits.  The RoPE frequencies go to the kernel as
 * parameters.
 *
 * Rules:
 *   - n <= RC_NOALLOC_MAX_TOKENS, else RC_ERR_ARG (nothing is launched).
 *   - The first call on a device looks up the array's device address on the
 *     current device (cudaGetSymbolAddress) and keeps it; make that first call
 *     before any stream capture.  Resetting that device (cudaDeviceReset)
 *     afterwards is not supported: the kept address would be stale.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents.  Calls that overlap on the GPU (other streams or
 *     threads without ordering) race on it; order them on one stream.
 *   - positions is a HOST array.  An arithmetic run p0, p0+1, ... needs no
 *     copy; any other position vector is copied into the array from the
 *     caller's (pageable) memory with cudaMemcpyAsync, which returns once the
 *     bytes are staged.
 *   - The caller keeps the ring state: delta_total (the sum of resets applied
 *     to this ring) and a write-group index in [0, slots) unique among the
 *     ring's live groups.  There is no delta rotation or attention entry on a
 *     caller-owned ring; this is the write alone.
 *
 * Ring layout (T = ceil(slots / 128) tiles per head, Cpad = 128 T), all device
 * memory the caller allocated:
 *   kcodes [heads][T][128][head_dim] E4M3: slot s is row s % 128 of tile
 *          s / 128; byte d of a row sits at 16-byte chunk (d / 16) XOR x,
 *          x = row % 8 (head_dim 128) or (row / 2) % 4 (head_dim 64).
 *   vcodes [heads][T][head_dim][128] E4M3 (transposed): element (d, s) sits in
 *          row d of tile s / 128 at chunk ((s % 128) / 16) XOR (d % 8).
 *   kscale, vscale [heads][Cpad] fp32: the scale of each slot's write group.
 *   group  [Cpad] int32: the slot's write-group index (-1 = empty).
 */
#define RC_NOALLOC_MAX_TOKENS 4096

typedef struct rc_ring_view {
    uint8_t *kcodes;  /* device, see the layout above */
    uint8_t *vcodes;
    float *kscale;
    float *vscale;
    int32_t *group;
    int heads;        /* >= 1 */
    int head_dim;     /* 64 or 128 */
    int slots;        /* ring capacity C >= 1 */
} rc_ring_view;

int rc_ring_write_noalloc(const rc_ring_view *ring, const void *K_bf16, const void *V_bf16,
                          const int64_t *positions, int n, int64_t delta_total,
                          int32_t group, double rope_base, void *stream);

/* Number of occupied slots of `layer`, or a negative status. */
int rc_cache_occupancy(const rc_cache *h, int layer);

/* Sum of all deltas applied so far. */
int64_t rc_cache_delta_total(const rc_cache *h);

/* Number of kernel launches this handle has made (for launch accounting). */
int64_t rc_cache_launch_count(const rc_cache *h);

/*
 * How the attention call treats the KV tiles of one ring (host only: no
 * device, no handle).  grp[0 .. slots) is the ring's write group per slot
 * (-1 = empty); tile t covers slots [128 t, min(128 t + 128, slots)).
 *   uniform[t / 64] bit t % 64: every slot of tile t holds the same write
 *     group, so one K and one V scale per head cover it (the fast path);
 *   split[t] = b in 1..127: tile t has 128 slots, [128 t, 128 t + b) hold one
 *     write group and [128 t + b, 128 t + 128) another (where a write's run of
 *     slots ends inside the tile; the two-run path); otherwise 0.
 * Every other tile takes the general path (per-slot scales and validity).
 * uniform (4 words) and split (256 bytes) are caller-owned host memory.
 * Errors: RC_ERR_ARG if a pointer is NULL or slots is outside 1 .. 32768.
 */
int rc_tile_kinds(const int32_t *grp, int slots, uint64_t *uniform, uint8_t *split);

#ifdef __cplusplus
}
#endif

#endif /* RC_H */
