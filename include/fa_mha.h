/*
 * fa_mha.h -- C ABI of the GB300 (sm_103a) fused multi-head attention forward,
 * without KV cache (fa_mha_no_cache*) and over a KV cache (fa_mha_kv_cache).
 *
 * The operation is the `mo.mha.no_cache` operator documented on the MAX API
 * page "FlashAttentionGPU" (method `execute`, Steps -1 to 4, and its
 * Parameters / Args lists):
 *
 *   out[b,i,h,:] = sum_j softmax_j( mask( scale * q[b,i,h,:] . k[b,j,hk,:] ) ) v[b,j,hk,:]
 *
 * with q, k, v and out in BSHD layout (the transposes of Step 0 and Step 4 are
 * folded into the kernel's addressing), grouped-query attention when k/v
 * carry Hkv < H heads (BShD; query head h reads KV head hk = h / (H / Hkv),
 * i.e. consecutive query heads share a KV head), and a mask that is none,
 * causal (key j visible to query i iff j <= i), causal with a sliding window
 * of W keys (visible iff j <= i and i - j < W), or a two-sided window without
 * the causal mask (visible iff |i - j| < W). The S x S score matrix
 * is never materialised: the bf16 path is a FlashAttention-2 style kernel
 * (online softmax over KV tiles, one final division by the running sum) on
 * the sm_103a tensor cores.
 *
 * Every buffer is owned by the caller. All entry points are plain C; device
 * pointers are CUDA device addresses on the current device, `stream` is a
 * cudaStream_t passed as void* (NULL = legacy default stream).
 */
#ifndef FA_MHA_H_
#define FA_MHA_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Mask kinds (the page's `mask_str`, chosen at run time here). */
#define FA_MASK_NONE 0
#define FA_MASK_CAUSAL 1

/* Element types of q, k, v and out (all four share one type). */
#define FA_DTYPE_BF16 0 /* tensor-core path, fp32 accumulation, bf16 output */
#define FA_DTYPE_F32 1  /* CUDA-core fp32 path (exact fp32 FMA arithmetic) */

/* Status codes returned by every entry point. */
typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* a null pointer, a bad size, a bad mask/window */
  FA_ERR_UNSUPPORTED = 2, /* valid but not built: D, dtype, GPU arch, alignment */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 4,     /* a kernel gave up on a bounded wait (see fa_stream_status) */
  FA_ERR_BOUNDS = 5       /* debug build only: a bounds guard skipped an out-of-range access */
} fa_status_t;

/*
 * fa_mha_no_cache -- the fused attention forward (FlashAttentionGPU.execute).
 *
 *   out   : device, [B, S, H, D], same dtype as q (the page: "same shape as q").
 *   lse   : device, [B, H, S] fp32, or NULL. Per query row the natural-log
 *           log-sum-exp of the scaled, masked scores (not on the pages; the
 *           statistic a split-KV combine consumes).
 *   q     : device, [B, S, H, D] (BSHD).
 *   k, v  : device, [B, S, Hkv, D] (BSHD when Hkv == H, BShD otherwise).
 *   B, S, H, Hkv, D : sizes; B, S, H, Hkv >= 1, H % Hkv == 0. D: for
 *           FA_DTYPE_BF16 a multiple of 8 up to 256 (the kernels work on 64,
 *           128 or 256 columns; TMA zero-fills the rest and clips it on store;
 *           above 128 also H / Hkv <= 128), for FA_DTYPE_F32 one of 32, 64, 96,
 *           128.
 *   scale : multiplies q.k before masking and softmax (the page's `scale`);
 *           finite and >= 0.
 *   mask_kind : FA_MASK_NONE or FA_MASK_CAUSAL.
 *   local_window_size : -1 for no window, else W >= 1: with FA_MASK_CAUSAL
 *           query i sees keys i-W+1 .. i, with FA_MASK_NONE keys i-W+1 ..
 *           i+W-1 (W >= S hides nothing).
 *   dtype : FA_DTYPE_BF16 or FA_DTYPE_F32.
 *   stream: cudaStream_t (as void*) the work is enqueued on.
 *
 * Layout: dense and contiguous, D fastest. bf16 buffers must be 16-byte
 * aligned (the kernel reads them with TMA). Sizes must keep every tensor
 * below 2^31 elements per dimension product used in indexing (checked).
 *
 * Behaviour: asynchronous on `stream`; returns after validation and launch.
 * Argument errors return FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED before any
 * CUDA call. A kernel that exceeds its bounded-wait limit abandons its tile,
 * sets the sticky status word of `stream` and leaves the outputs of that
 * tile undefined; read it with fa_stream_status(stream) (ordered on that
 * stream only) or fa_device_status() (every stream of a device).
 *
 * Per-device state, created lazily and freed by fa_shutdown(): the first
 * call on a device allocates that device's status words (one 4 KB cudaMalloc)
 * and raises each kernel's shared-memory limit once; the TMA tensor maps of
 * a call are cached, keyed on address, sizes and strides, so a repeated call
 * on the same buffers encodes nothing. Make the first call on a device before
 * any stream capture. Thread-safe.
 */
fa_status_t fa_mha_no_cache(void *out, float *lse, const void *q, const void *k, const void *v,
                            int B, int S, int H, int Hkv, int D, float scale, int mask_kind,
                            int local_window_size, int dtype, void *stream);

/*
 * fa_mha_no_cache_strided -- fa_mha_no_cache on strided views: each of q, k,
 * v and out may be any BSHD view whose D dimension is contiguous, e.g. slices
 * of a packed [B, S, H + 2 Hkv, D] QKV projection, or a [B, H, S, D] tensor
 * viewed as BSHD (the Step 0 / Step 4 transposes of the FlashAttentionGPU
 * page then cost nothing: the kernels address the views directly).
 *
 *   x_strides : 3 element strides of that tensor along B, S and H (all >= 1;
 *               for FA_DTYPE_BF16 multiples of 8 elements, i.e. 16 bytes, as
 *               TMA requires).
 * Every other argument, the lse layout ([B, H, S], dense) and the behaviour
 * are those of fa_mha_no_cache. out must not overlap q, k or v.
 */
fa_status_t fa_mha_no_cache_strided(void *out, float *lse, const void *q, const void *k,
                                    const void *v, int B, int S, int H, int Hkv, int D,
                                    const long long *q_strides, const long long *k_strides,
                                    const long long *v_strides, const long long *out_strides,
                                    float scale, int mask_kind, int local_window_size, int dtype,
                                    void *stream);

/*
 * fa_mha_no_cache_noalloc -- the same bf16 attention forward as
 * fa_mha_no_cache, for callers that cannot allocate device memory. The pages
 * describe nothing like it; it exists for code that does not own the CUDA
 * allocator (a framework's caching allocator or a pool sized up front),
 * must not allocate on a latency-critical path, or must account for every
 * allocation before it starts.
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine. The one
 * piece of global memory the kernel needs besides its inputs and outputs (a
 * 4-byte status word) lives in a 256-byte array inside this library that
 * every GPU loading the library holds until the process exits; sizes that
 * would need more scratch than that are rejected with FA_ERR_UNSUPPORTED
 * (the status word does not grow with B, S, H or D, so no size is).
 *
 * Arguments are those of fa_mha_no_cache for dtype FA_DTYPE_BF16 (the only
 * dtype it takes) with D a multiple of 8 up to 128 (the head dims of the
 * prefill kernel; larger ones are rejected with FA_ERR_UNSUPPORTED), plus
 * check_status: when non-zero the call synchronises `stream` after the
 * launch and returns FA_ERR_TIMEOUT if the kernel gave up on a bounded wait
 * (the limit set by fa_set_wait_timeout_ns); when zero it returns right after
 * the launch, and a time-out is then reported nowhere: the outputs of the
 * abandoned tiles are undefined and the next call clears the word. Each call
 * clears the status word on `stream` before its launch. The word is not one
 * of the words fa_stream_status and fa_device_status read.
 *
 * The first call on each device resolves the array's device address (a
 * cudaGetSymbolAddress set-up step); make that first call before any stream
 * capture. All calls share the one array: calls that overlap on the GPU (on
 * different streams) race on the status word, so one call may report or hide
 * another's time-out.
 */
fa_status_t fa_mha_no_cache_noalloc(void *out, float *lse, const void *q, const void *k,
                                    const void *v, int B, int S, int H, int Hkv, int D,
                                    float scale, int mask_kind, int local_window_size,
                                    void *stream, int check_status);

/*
 * fa_mha_no_cache_host -- fa_mha_no_cache with q, k, v, out and lse in HOST
 * memory: enqueues on `stream` the copies of q, k and v into `workspace`, the
 * forward, and the copies of out (and lse) back to the host. Returns after
 * enqueueing; the host outputs are complete once `stream` has been
 * synchronised. With page-locked (pinned) host buffers every copy is
 * asynchronous, so calls alternating over two streams (each with its own
 * workspace) overlap one call's copies with the other's kernel; with
 * pageable buffers CUDA performs the copies synchronously.
 *
 *   out, lse, q, k, v : host, layouts as fa_mha_no_cache (dense); lse may be
 *             NULL.
 *   workspace, workspace_bytes : caller-owned device buffer of at least
 *             fa_mha_no_cache_host_workspace(B, S, H, Hkv, D, dtype) bytes,
 *             256-byte aligned; it receives the device copies of q, k, v,
 *             out and lse (and, for fp32 with D 64 or 128, the bf16 parts of
 *             K and V: that case runs on the tensor cores as
 *             fa_mha_no_cache_f32_tc).
 * Every other argument, and the error behaviour, as fa_mha_no_cache; all
 * arguments are checked before the first copy is enqueued.
 */
fa_status_t fa_mha_no_cache_host(void *out, float *lse, const void *q, const void *k,
                                 const void *v, int B, int S, int H, int Hkv, int D, float scale,
                                 int mask_kind, int local_window_size, int dtype, void *workspace,
                                 unsigned long long workspace_bytes, void *stream);

/* Device bytes fa_mha_no_cache_host needs (0 for sizes below 1 or a bad dtype). */
unsigned long long fa_mha_no_cache_host_workspace(int B, int S, int H, int Hkv, int D, int dtype);

/*
 * fa_mha_no_cache_f32_tc -- fa_mha_no_cache for fp32 tensors on the tensor
 * cores at fp32 accuracy (the page's `scale: Float32` interface with fp32
 * q, k, v): every operand is split into three bf16 parts (x = b0 + b1 + b2,
 * 24 significant bits) and each contraction sums the six part products down
 * to 2^-16 of the leading one, with fp32 accumulation; max-abs error on the
 * bench workloads stays within 1e-4 of the exact result, like the CUDA-core
 * fp32 path (FA_DTYPE_F32 of fa_mha_no_cache).
 *
 *   out, lse, q, k, v, sizes, scale, mask_kind, local_window_size : as
 *             fa_mha_no_cache with fp32 data, dense BSHD / BShD, 16-byte
 *             aligned; D in {64, 128}; finite inputs.
 *   workspace, workspace_bytes : caller-owned device scratch of at least
 *             fa_mha_no_cache_f32_tc_workspace(B, S, Hkv, D) bytes (K's and
 *             V's bf16 planes), 256-byte aligned.
 * Asynchronous on `stream`; errors as fa_mha_no_cache.
 */
fa_status_t fa_mha_no_cache_f32_tc(float *out, float *lse, const float *q, const float *k,
                                   const float *v, int B, int S, int H, int Hkv, int D,
                                   float scale, int mask_kind, int local_window_size,
                                   void *workspace, unsigned long long workspace_bytes,
                                   void *stream);

/* Bytes of workspace fa_mha_no_cache_f32_tc needs (0 for unsupported sizes). */
unsigned long long fa_mha_no_cache_f32_tc_workspace(int B, int S, int Hkv, int D);

/*
 * fa_mha_kv_cache -- attention over a KV cache (bf16, tensor cores). The
 * pages document only the no-cache operator; this is its cached sibling read
 * the plain way: the same operator (FlashAttentionGPU.execute, Steps -1 to 4)
 * when the keys and values of batch b are the first L_b = cache_lens[b] rows
 * of a cache and the Sq queries are the last Sq tokens of that sequence, so
 * query row s sits at position L_b - Sq + s and the mask (causal: keys j <=
 * position; window W: position - j < W, or |position - j| < W without the
 * causal mask) is evaluated there. Sq = 1 is one decoding step; Sq > 1 covers
 * speculative or chunked steps.
 *
 *   out     : device, [B, Sq, H, D] bf16 (BSHD).
 *   lse     : device, [B, H, Sq] fp32, or NULL (natural log, scale included).
 *   q       : device, [B, Sq, H, D] bf16 (BSHD).
 *   k_cache, v_cache : device, [B, S_cache, Hkv, D] bf16 (BShD); rows at
 *             positions >= L_b are never used (they may hold anything).
 *   cache_lens : device, B int32 key counts (values outside [0, S_cache] are
 *             clamped into it), or NULL for S_cache keys in every batch.
 *   B, Sq, S_cache, H, Hkv, D : sizes; all >= 1, H % Hkv == 0,
 *             H / Hkv <= 128, D a multiple of 8 up to 256.
 *   scale, mask_kind, local_window_size : as fa_mha_no_cache.
 *   num_splits : 0 lets the library share out the work. A unit is one
 *             (batch, KV head, position tile of up to 128 / (H / Hkv)
 *             queries). Units that fill half the SMs run whole, one CTA each.
 *             Fewer units are shared out stream-K fashion: groups of Hkv
 *             persistent CTAs (one per KV head, 27/32 of the SMs in all)
 *             take equal contiguous quotas of all units' key tiles, found
 *             from cache_lens on the device, and a unit is cut where a quota
 *             ends. n >= 1 asks for n even key ranges per unit (capped at
 *             the number of key tiles and at 128), which persistent CTAs
 *             share round-robin. Cut units are merged by a second kernel.
 *   workspace, workspace_bytes : caller-owned device scratch of at least the
 *             size fa_mha_kv_cache_plan returns for the same arguments (may be
 *             NULL when that size is 0); 16-byte aligned.
 *   dtype   : FA_DTYPE_BF16 (the only type this entry point takes).
 *   stream  : cudaStream_t as void*.
 *
 * A query that sees no key (L_b = 0, or a causal row whose position L_b - Sq
 * + s is negative) gets out = 0 and lse = -inf. Behaviour on errors and
 * time-outs is that of fa_mha_no_cache.
 */
fa_status_t fa_mha_kv_cache(void *out, float *lse, const void *q, const void *k_cache,
                            const void *v_cache, const int *cache_lens, int B, int Sq,
                            int S_cache, int H, int Hkv, int D, float scale, int mask_kind,
                            int local_window_size, int num_splits, void *workspace,
                            unsigned long long workspace_bytes, int dtype, void *stream);

/*
 * fa_mha_kv_cache_plan -- how fa_mha_kv_cache will cut the work for these
 * arguments: *splits_out receives 1 when every unit runs whole, else the
 * most pieces one unit can be cut into (the requested ranges, or the number
 * of CTA groups of the stream-K plan); *workspace_bytes_out the scratch it
 * needs (0 when every unit runs whole: fp32 partial O rows and LSEs, one slot
 * of H / Hkv x (position-tile) rows per piece).
 * num_sms = 0 uses the current device's SM count (the one fa_mha_kv_cache
 * uses); n >= 1 plans for a device with n SMs and makes no CUDA call.
 */
fa_status_t fa_mha_kv_cache_plan(int B, int Sq, int S_cache, int H, int Hkv, int D, int mask_kind,
                                 int local_window_size, int num_splits, int num_sms,
                                 int *splits_out, unsigned long long *workspace_bytes_out);

/*
 * fa_topk -- exact top-K selection per row: the op of the Modular recipe
 * "Custom Operations: Applications in AI Models", section "Optimizing top-K
 * token sampling for GPUs in MAX" (each row of scores comes back ordered by
 * highest value, as values and indices). Order: descending IEEE-754 total
 * order (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN); equal values by
 * ascending index, so the result is unique.
 *
 *   values  : device, [B, K] fp32, written (descending).
 *   indices : device, [B, K] int32, written (column of each value in its row).
 *   scores  : device, [B, V] fp32, rows row_stride elements apart (>= V).
 *   B, V, K : 1 <= B <= 65535, V >= 1, 1 <= K <= min(V, 1024).
 *   workspace, workspace_bytes : caller-owned device scratch of at least the
 *             size fa_topk_plan returns for (B, V, K) (may be NULL when that
 *             size is 0: every row is one chunk); 8-byte aligned.
 *   stream  : cudaStream_t as void*.
 * Asynchronous; argument errors are returned before any CUDA call.
 */
fa_status_t fa_topk(float *values, int *indices, const float *scores, int B, int V,
                    long long row_stride, int K, void *workspace,
                    unsigned long long workspace_bytes, void *stream);

/*
 * fa_topk_plan -- chunks per row and workspace bytes fa_topk uses for (B, V,
 * K); num_sms = 0 plans for the current device, n >= 1 for an n-SM device
 * (no CUDA call).
 */
fa_status_t fa_topk_plan(int B, int V, int K, int num_sms, int *chunks_out,
                         unsigned long long *workspace_bytes_out);

/*
 * fa_stream_status -- the sticky status of the work this library enqueued on
 * `stream` (a cudaStream_t of the current device, as void*; NULL = legacy
 * default stream): FA_OK, FA_ERR_TIMEOUT if a kernel launched on that stream
 * since the last clear abandoned a bounded wait, or FA_ERR_BOUNDS (debug
 * build) if a bounds guard fired. The read is a copy ordered on `stream`
 * followed by cudaStreamSynchronize(stream): it waits for that stream's work
 * only, never for the device. With clear != 0 the word is reset (also on
 * `stream`). Each stream has its own word for the first 1023 streams used on
 * a device; later streams share one word. A stream handle that is destroyed
 * and re-created at the same address keeps the old stream's word until it is
 * cleared. Returns FA_ERR_CUDA if the copy or the synchronisation fails.
 */
fa_status_t fa_stream_status(void *stream, int clear);

/*
 * fa_device_status -- synchronises `device` (cudaDeviceSynchronize) and reads
 * the status words of all its streams: FA_OK, FA_ERR_TIMEOUT if any kernel
 * since the last clear abandoned a bounded wait, FA_ERR_BOUNDS (debug build)
 * if a bounds guard fired. With clear != 0 every word is reset. Returns
 * FA_ERR_CUDA if the synchronisation itself reports an error.
 */
fa_status_t fa_device_status(int device, int clear);

/*
 * fa_set_wait_timeout_ns -- limit, in nanoseconds of GPU global timer, of
 * every spin-wait inside the kernels (default 2e9). A value of 0 restores the
 * default. Affects launches made after the call. Returns the previous limit.
 */
unsigned long long fa_set_wait_timeout_ns(unsigned long long ns);

/*
 * fa_set_stall_probe -- test hook for the time-out path. While enabled, the
 * MMA-issuing thread of every bf16 launch first waits on a barrier that
 * nothing signals; that wait ends when the bounded-wait limit expires, so
 * every CTA takes its time-out path (records FA_ERR_TIMEOUT, drains its own
 * copies, frees tensor memory, returns) and the outputs are undefined. The
 * launch still completes and the context stays usable. Affects launches made
 * after the call; returns the previous setting (0 or 1).
 */
int fa_set_stall_probe(int enable);

/* fa_status_string -- a static, human-readable name for a status code. */
const char *fa_status_string(fa_status_t status);

/*
 * fa_last_error_message -- detail of the last non-OK status returned on the
 * calling thread (which argument was rejected, which CUDA call failed).
 * The string is owned by the library and valid until the next call.
 */
const char *fa_last_error_message(void);

/* fa_version -- library version as major*10000 + minor*100 + patch. */
int fa_version(void);

/*
 * fa_trace_set_buffer -- debug build (libfa_mha_debug.so, compiled with
 * FA_TRACE=1) only: record an event trace of every later launch of the
 * bf16 prefill kernel (D <= 128) into `buf`, a caller-owned, 16-byte-aligned
 * device buffer of `bytes` bytes: fa_trace_bytes_per_cta() bytes for each
 * CTA, CTA c at offset c * fa_trace_bytes_per_cta(); CTAs past the buffer
 * record nothing. Each CTA holds 10 roles (TMA producer, MMA issuer, softmax
 * warps 0 and 4 -- the first of Q tile 0 and of Q tile 1 -- then softmax
 * warps 1, 2, 3, 5, 6, 7) x 256 records of 16 bytes: global timer
 * in ns (two 32-bit words), the SM's clock (low 32 bits), and event code <<
 * 24 | 24-bit argument; the codes are listed in csrc/fa_trace.cuh. A role's
 * records past 256 are dropped; records not written are left as they were
 * (zero the buffer first). NULL stops tracing. The default build returns
 * FA_ERR_UNSUPPORTED (and FA_OK for NULL).
 */
fa_status_t fa_trace_set_buffer(void *buf, unsigned long long bytes);

/* fa_trace_bytes_per_cta -- trace bytes per CTA (0 in the default build). */
unsigned long long fa_trace_bytes_per_cta(void);

/*
 * fa_trace_ctas -- CTAs of one bf16 prefill launch of the debug build
 * (D <= 128) for these sizes: one per (query block, head, batch), blocks of
 * 128 queries for D up to 64, else of 256; 0 for sizes that launch another
 * kernel. (The default build runs head dims up to 64 on a persistent grid of
 * at most two CTAs per SM instead.)
 */
long long fa_trace_ctas(int B, int S, int H, int D);

/*
 * fa_debug_set_lse_limit -- debug build only: the number of LSE elements the
 * prefill kernel's bounds guard lets it write (0: all B * H * S). Elements
 * past the limit are skipped and the stream's status reports FA_ERR_BOUNDS.
 * Exists to test that the guards fire; the default build returns
 * FA_ERR_UNSUPPORTED.
 */
fa_status_t fa_debug_set_lse_limit(long long elems);

/*
 * fa_shutdown -- frees the per-device status words and empties the tensor-map
 * cache. Call only when no work issued by this library is pending; later
 * calls re-create what they need.
 */
void fa_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_MHA_H_ */
