/*
 * moe.h - C ABI of the decode-time routed Mixture-of-Experts layer (GB300, sm_103a).
 *
 * One context holds one stack of MoE layers: a router per layer, the routed experts
 * stored in a low-bit format, and an optional always-on shared expert.  For every
 * token the layer
 *   1. runs the router GEMV  logit[e] = sum_h x[h] * W_r[e,h]  (fp32),
 *   2. picks the top-k experts by logit (equal logits: the lower expert id first) and
 *      weights them, either softmax renormalised over the k selected, or sigmoid
 *      scores divided by their sum over the k selected,
 *   3. applies only the selected experts' SwiGLU FFN  y_e = W_d (silu(W_g x) * (W_u x)),
 *      dequantising their low-bit weights on the fly,
 *   4. combines  out = sum_j w_j y_{e_j}  in rank order, then adds the shared expert.
 * Sources: "WISP - streaming what can't run" (molayo1419.me), section "Insight
 * (Credit: JustVugg / Colibri)": the model's own router picks the experts of each
 * token, and only those are fetched; section "Lesson 2: the model's router is the
 * best scheduler".  "Introducing WARP" (discuss.pytorch.kr), section "The paradox in
 * WARP's cache settings": num_experts_per_token (k) is a parameter of the model.
 *
 * Expert weights (boundary blob formats, little-endian, one contiguous record per
 * expert: "2.78T-parameter model on a laptop: the NVMe streaming inference engine
 * WASTE" (ttj.ttj.kr), section "Idle weights only need to arrive on time": each
 * expert record holds gate, up and down adjacent so one read fetches an expert; the
 * experts are residual-vector-quantised at 3.00 bits per weight and never expanded):
 *
 *   MOE_W_RVQ3_G8: for each matrix in the order gate [F,H], up [F,H], down [H,F]
 *     (rows x K, K = the input dimension):
 *       fp16 codebooks [3][256][8]  (stage 0, 1, 2),
 *       uint8 codes    [rows][K/8][3] (stage order 0, 1, 2 within a group),
 *     and W[r, 8q+i] = C0[c0][i] + C1[c1][i] + C2[c2][i].  K must be a multiple of 8.
 *   MOE_W_INT4_G128: for each matrix in the same order:
 *       uint8 nibbles [rows][K/2] (low nibble = even input index; two's complement
 *       q in [-8, 7]), then fp16 scales [rows][K/128]; W[r,k] = q[r,k] * s[r,k/128].
 *     K must be a multiple of 128.
 *
 * Experts live either all resident in HBM (hbm_cache_bytes == 0) or in a pinned host
 * pool with a bounded HBM LRU cache filled on a miss over a side stream ("WISP",
 * sections "Insight" (VRAM -> RAM -> SSD lookup with LRU promotion) and
 * "Double-Buffer Async Pipeline"; "WASTE", section "Idle weights only need to arrive
 * on time": the remaining memory is a bounded expert cache).  Caching changes timing,
 * never results ("Introducing WARP", section "How WARP keeps the model out of RAM").
 *
 * Conventions shared by every call:
 *   - Return MOE_OK or an error; nothing is thrown.  Argument errors are reported at
 *     once and leave the context unchanged.
 *   - Asynchronous CUDA failures and device wait time-outs are sticky: once seen, every
 *     later call on the context returns MOE_ECUDA or MOE_ETIMEOUT until moe_destroy.
 *   - Host pointers are copied during the call; the caller may free them on return.
 *   - Device pointers (x, out) belong to the caller and must stay valid until the
 *     stream has run the call.
 *   - A context is single-threaded.  All forwards on one context must be ordered on
 *     the device (one stream, or streams the caller orders), because they share the
 *     context's scratch buffers.
 *   - "stream" is a cudaStream_t passed as void* (NULL = the legacy default stream).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_EINVAL = 1,     /* bad argument (null, out of range, size mismatch) */
    MOE_ENOMEM = 2,     /* HBM or pinned host memory could not be allocated */
    MOE_EBUDGET = 3,    /* the HBM cache cannot hold one layer's working set
                           (max(2 k, min(E, max_tokens k)) records) */
    MOE_ECUDA = 4,      /* a CUDA call failed (sticky) */
    MOE_ESTATE = 5,     /* a router or expert of the layer is not registered yet */
    MOE_ETIMEOUT = 6,   /* a bounded device wait ran out (sticky) */
    MOE_ENOTFOUND = 7,  /* nothing recorded yet (moe_get_routing before a forward) */
    MOE_EIO = 8         /* the expert file could not be created, written or read */
} moe_status;

typedef enum {
    MOE_ROUTER_SOFTMAX_TOPK_RENORM = 0, /* w = softmax of the k selected logits */
    MOE_ROUTER_SIGMOID_TOPK_NORM = 1    /* w = sigmoid(l_j) / sum_sel sigmoid(l) */
} moe_router;

typedef enum {
    MOE_W_RVQ3_G8 = 1,   /* 3 x uint8 codes per 8 weights, 3 fp16 256x8 codebooks per matrix */
    MOE_W_INT4_G128 = 2  /* symmetric int4, fp16 scale per 128 input elements */
} moe_wfmt;

typedef struct {
    int num_layers;     /* >= 1 */
    int hidden;         /* H */
    int ffn;            /* F of every routed expert */
    int num_experts;    /* E routed experts per layer, 1..1024 */
    int top_k;          /* k, 1..min(E, 32) */
    int shared_ffn;     /* 0 = no shared expert, else must equal ffn */
    int router;         /* moe_router */
    int wfmt;           /* moe_wfmt */
    int max_tokens;     /* largest T of a forward, 1..256 */
    unsigned long long hbm_cache_bytes; /* 0 = every expert resident in HBM; else the
                                           HBM budget of the expert cache in bytes */
    const char* pool_file;              /* streamed mode: NULL = the host pool holds every
                                           expert in pinned RAM; else the experts live in this
                                           file (created, truncated, removed by moe_destroy)
                                           behind a pinned RAM cache of host_cache_bytes;
                                           read by MOE_FILE_READERS threads (env, 1..64,
                                           default 8) */
    unsigned long long host_cache_bytes; /* with pool_file: the RAM cache budget in bytes
                                            (at least 2 k records of 4096-byte aligned size) */
} moe_config;

typedef struct {
    unsigned long long forwards;              /* moe_forward calls that ran */
    unsigned long long tokens;                /* sum of T over those calls */
    unsigned long long lookups;               /* one per (layer, forward, unique expert) */
    unsigned long long hits;                  /* lookups served from HBM */
    unsigned long long misses;                /* lookups copied from the host pool */
    unsigned long long bytes_expert_touched;  /* kernel-layout record bytes of the unique
                                                 experts of each forward (incl. shared) */
    unsigned long long bytes_router;          /* router weight bytes read */
    unsigned long long bytes_h2d;             /* expert bytes copied host -> device */
    unsigned long long record_bytes;          /* kernel-layout bytes of one expert */
    unsigned long long cache_slots;           /* HBM expert slots (0 when all resident) */
    double h2d_ms;                            /* time the host->device link was busy with expert
                                                 copies: the union over copy batches (one
                                                 forward's misses, or one read-ahead) of first
                                                 copy start to last copy end (streamed) */
    unsigned long long prefetches;            /* records copied by read-ahead (streamed) */
    unsigned long long prefetch_hits;         /* lookups that found a record read-ahead put there
                                                 and no lookup had used yet */
    unsigned long long file_reads;            /* records read from the expert file (pool_file) */
    unsigned long long file_read_bytes;       /* bytes of those reads (4096-byte aligned records) */
    unsigned long long ram_hits;              /* HBM misses served from the RAM cache (pool_file) */
    unsigned long long ram_misses;            /* HBM misses read from the file first (pool_file) */
    double file_read_ms;                      /* wall time of the file read batches */
    int file_direct;                          /* 1 when the file is read with O_DIRECT */
    unsigned long long launches;              /* kernels launched by the forward calls (counted on
                                                 the host when the call queues them; calls recorded
                                                 into a CUDA graph count once, at capture) */
} moe_stats_t;

typedef struct moe_ctx moe_ctx;

/* Create a context on CUDA device `device`.  Allocates the HBM expert storage (all
 * experts when hbm_cache_bytes == 0, else floor(hbm_cache_bytes / record) slots),
 * the pinned host pool (streamed mode only: every expert, or with pool_file the RAM
 * cache in front of the expert file), router storage and scratch.
 * Errors: MOE_EINVAL (bad config; pool_file without hbm_cache_bytes), MOE_EBUDGET (HBM
 * cache below max(2 k, min(E, max_tokens k)) records, a forward's worst-case working set
 * beside the next layer's; above what the pool needs is allowed and clipped; RAM cache
 * below 2 k records), MOE_ENOMEM (HBM or host memory short; checked against
 * cudaMemGetInfo before allocating), MOE_EIO (the expert file), MOE_ECUDA. */
moe_status moe_create(const moe_config* cfg, int device, moe_ctx** out);

/* Register the router of `layer`: fp32 [E][H] row-major.  `w` may be host memory or
 * device memory of the context's device; it is copied. */
moe_status moe_register_router(moe_ctx* ctx, int layer, const float* w);

/* Register expert `expert` (0..E-1, or -1 for the shared expert) of `layer` from its
 * boundary blob (format above).  `blob` may be host memory or device memory of the
 * context's device; `bytes` must equal moe_expert_blob_bytes().  The blob is repacked
 * into the kernel layout: into its HBM slot (resident mode), into the pinned host pool
 * (streamed mode) or into the expert file (pool_file).  Synchronous: the blob may be freed
 * on return.  MOE_EIO when the file write fails. */
moe_status moe_register_expert(moe_ctx* ctx, int layer, int expert, const void* blob, size_t bytes);

/* Size in bytes of one expert blob in the boundary format, or 0 for a bad shape. */
size_t moe_expert_blob_bytes(int wfmt, int hidden, int ffn);

/* One MoE layer on T tokens: out[T,H] (fp32) = combine of the routed experts (+ shared)
 * applied to x[T,H] (bf16 bits, row-major).  x and out are device pointers, x 16-byte
 * aligned.
 * Resident mode: fully stream-ordered, never blocks the host, capturable in a CUDA
 * graph.  Streamed mode: blocks the host once per call to read the routing back, then
 * issues the miss copies on a side stream, hits first, each missed expert's kernels
 * waiting for its own copy.  Errors: MOE_EINVAL (T outside 1..max_tokens, layer out of
 * range, null pointers), MOE_ESTATE (layer not fully registered), sticky errors.
 * Numerics: the int4 kernels, and the RVQ down projection, carry their activations as fp16
 * hi + lo pairs (their sum equals the fp32 value to 2^-22 of it), so the input x and the
 * SwiGLU activations silu(W_g x) * (W_u x) must stay below 65504 in magnitude; sums are
 * fp32 and the output is fp32. */
moe_status moe_forward(moe_ctx* ctx, int layer, const void* x_bf16, float* out, int T, void* stream);

/* One layer of the residual stack, fused:  if y_prev != NULL: x += y_prev;
 * xn = bf16(x / sqrt(mean(x^2) + eps));  y = layer(xn)  (as moe_forward).
 * x fp32 [T,H] in/out, y_prev fp32 [T,H] or NULL (it may be the same buffer as y),
 * xn bf16 bits [T,H] out, y fp32 [T,H] out; all device pointers, x, y_prev and xn 16-byte
 * aligned (MOE_EINVAL otherwise).  Same bits as
 * moe_residual_rmsnorm followed by moe_forward; for small T the norm runs inside the
 * router kernel instead of a kernel of its own. */
moe_status moe_forward_residual(moe_ctx* ctx, int layer, float* x, const float* y_prev, uint16_t* xn,
                                float* y, int T, float eps, void* stream);

/* The routing of the last forward of `layer`: idx[T][k] (int32, descending score) and
 * w[T][k] (fp32) into host buffers; *T_out = that forward's T.  Synchronises the device.
 * MOE_ENOTFOUND before the first forward of the layer. */
moe_status moe_get_routing(moe_ctx* ctx, int layer, int* idx, float* w, int* T_out);

/* Residual + RMS norm of the stack that feeds one layer into the next:
 *   if y != NULL: x += y;   xn = bf16(x / sqrt(mean(x^2) + eps))   (no gain),
 * on T rows of H = the context's hidden size; x fp32 [T,H] in/out, y fp32 [T,H],
 * xn bf16 bits [T,H], all device pointers (x, y 16-byte aligned), stream-ordered. */
moe_status moe_residual_rmsnorm(moe_ctx* ctx, float* x, const float* y, uint16_t* xn, int T,
                                float eps, void* stream);

/* Counters since create (or the last reset).  Also surfaces sticky asynchronous errors
 * (it synchronises the context's device). */
moe_status moe_stats(moe_ctx* ctx, moe_stats_t* out);
moe_status moe_reset_stats(moe_ctx* ctx);

/* Read-ahead (streamed contexts; "Introducing WARP", section How WARP keeps the model out
 * of RAM: predict the next layer's experts and start loading them early).  With enable = 1,
 * every moe_forward / moe_forward_residual of layer l < num_layers - 1 ends by applying
 * layer l+1's router to layer l's router input (bf16 xn) with its own scratch, reading the
 * predicted experts back (the host waits for that small router only), and queuing copies
 * of the predicted experts that are not cached into least-recently-used unpinned slots,
 * behind layer l's miss copies.  The next forward finds them as hits; its kernels for such
 * an expert wait for that copy.  Results are bit-identical with and without read-ahead;
 * a wrong prediction only costs link time.  Meant for callers that run the layers in
 * order.  enable = 0 turns it off (the default).  MOE_EINVAL for enable outside {0, 1}, or
 * enable = 1 on a context with every expert resident. */
moe_status moe_set_readahead(moe_ctx* ctx, int enable);

/* Release everything the context owns.  Safe on NULL. */
moe_status moe_destroy(moe_ctx* ctx);

const char* moe_strerror(moe_status s);

/* Routing of T tokens without allocating anything (no counterpart in the pages).
 * For callers that cannot allocate device memory when they route: code recording a CUDA
 * graph (cudaMalloc is not allowed during stream capture), an engine whose own memory
 * pool already holds the free device memory, or a host application whose plugin rules
 * forbid allocation.  It runs the router of moe_forward (router GEMV, top-k, softmax
 * renormalised or sigmoid normalised weights) on x bf16 [T,H] with W fp32 [E,H] (device
 * pointers, x 8-byte and W 16-byte aligned, no context needed) and writes idx int32
 * [T,k] and w fp32 [T,k] (device) on
 * `stream`, the same values moe_forward records for moe_get_routing.
 * Scratch: one 1 MiB device array per device, held for the life of the process; calls
 * whose partial logits ((ceil(H/1024) + 1) * T * E floats) and plan do not fit return
 * MOE_EINVAL.  Limits otherwise as moe_config (T <= 256, E <= 1024, k <= 32, H % 8 == 0).
 * The first call on a device sets that device up (looks up the array's device address
 * and the kernel's shared-memory limit); make it before any stream capture.  Every call
 * shares the array and it keeps the last call's contents (the tickets it needs at zero
 * are cleared by each call on its stream), so calls that overlap on the GPU (different
 * streams, or other threads) race: order them.  Uses the current device. */
moe_status moe_route_noalloc(const uint16_t* x_bf16, const float* W, int T, int H, int E, int k, int router,
                             int* idx, float* w, void* stream);

/* ---- measurement (no counterpart in the pages) ---- */

/* Per-kernel timing: when enabled, moe_forward records CUDA events (timing enabled) on its
 * stream before the router and after the router, gate/up, down and combine kernels of
 * each layer (inside a CUDA graph capture they become event nodes of the graph).
 * moe_profile_read synchronises the device and returns, summed over the layers whose
 * latest forward was recorded, the milliseconds of [router, gate/up, down, combine] in
 * ms[0..3], and that number of layers in *n_layers.  Resident mode only. */
moe_status moe_profile(moe_ctx* ctx, int enable);
moe_status moe_profile_read(moe_ctx* ctx, double* ms, int* n_layers);

/* Work split of the RVQ lookup kernel (host code, no device): for u_n units of ntask
 * 32-row tasks over `grid` blocks with grid < u_n < 2 grid (a unit = one pass, matrix and
 * 512-input k-slice, each costing a table build), writes block b's task range
 * [t0[b], t1[b]) for b < grid, the same ranges the kernel's blocks take: groups of blocks
 * holding whole units, split greedily at rounds of 16 tasks, chosen for the least largest
 * block cost.  Returns 0, or 1 (nothing written) when u_n is outside (grid, 2 grid),
 * ntask or grid is not positive, u_n * ntask overflows an int or an array is null.  The
 * caller owns t0 and t1 (grid ints each). */
int moe_rvq_block_split(int u_n, int ntask, int grid, int* t0, int* t1);

/* ---- test hooks (no counterpart in the pages; failure injection on the host) ---- */

/* Make the next `n` host-to-device miss copies fail as if cudaMemcpyAsync had
 * returned an error; the forward then fails with the sticky MOE_ECUDA. */
moe_status moe_debug_fail_copies(moe_ctx* ctx, int n);

/* Run one bounded device wait on a flag that nothing sets, with a budget of `cycles`
 * SM clock cycles, on `stream`, and report the status word it leaves: MOE_ETIMEOUT is
 * the expected answer.  The time-out is recorded in *status only; it does not make the
 * context sticky. */
moe_status moe_debug_wait_timeout(moe_ctx* ctx, unsigned long long cycles, void* stream, int* status);

/* ---------------------------------------------------------------- the file tier alone
 * The RAM + file part of the streamed store on its own ("WISP - streaming what can't run",
 * section "Insight (Credit: JustVugg / Colibri)": VRAM, then RAM, then SSD, with LRU
 * promotion), host code only, for host-side tests and tools.  A context created with
 * moe_config.pool_file uses the same component with pinned RAM slots.
 * Records of rec_bytes are stored at key * stride, stride = rec_bytes rounded up to 4096;
 * keys are 0..n_keys-1.  The RAM cache holds floor(ram_bytes / stride) records (at most
 * n_keys), least recently used evicted first.  Reads of one fetch run on MOE_FILE_READERS
 * reader threads (env, 1..64, default 8), with O_DIRECT where the filesystem allows
 * (moe_filetier_info says which). */
typedef struct moe_filetier moe_filetier;
typedef struct {
    unsigned long long slots;       /* RAM cache records */
    unsigned long long stride;      /* bytes per record in the file and in RAM */
    int direct;                     /* 1 = O_DIRECT */
    unsigned long long reads;       /* records read from the file */
    unsigned long long read_bytes;
    unsigned long long ram_hits;    /* fetched keys found in RAM */
    unsigned long long ram_misses;  /* fetched keys read from the file */
    double read_ms;                 /* wall time of the read batches */
} moe_filetier_stats_t;

/* Create (truncate) the file `path` for n_keys records and allocate the RAM cache.
 * Errors: MOE_EINVAL, MOE_EBUDGET (ram_bytes below one record), MOE_ENOMEM, MOE_EIO. */
moe_status moe_filetier_create(const char* path, size_t rec_bytes, long long n_keys,
                               unsigned long long ram_bytes, moe_filetier** out);
/* Write record `key` (rec_bytes from `rec`, host memory).  A RAM copy of the key is
 * dropped.  Errors: MOE_EINVAL (bad key, nulls), MOE_EIO. */
moe_status moe_filetier_write(moe_filetier* ft, long long key, const void* rec);
/* Make n distinct keys resident in RAM (n <= slots) and return their RAM addresses in
 * out[n] and slots in slots[n]; they become the most recently used.  The addresses stay
 * valid until a later fetch or write.  Errors: MOE_EINVAL (n > slots, bad or duplicate
 * use), MOE_EIO (a read failed; out[] is NULL then). */
moe_status moe_filetier_fetch(moe_filetier* ft, const long long* keys, int n, const void** out, int* slots);
moe_status moe_filetier_info(const moe_filetier* ft, moe_filetier_stats_t* out);
/* Close and free (the file stays; the caller removes it). */
void moe_filetier_destroy(moe_filetier* ft);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
