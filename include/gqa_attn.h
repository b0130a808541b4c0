/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) causal grouped-query attention library.
 *
 * The library computes the attention of a hybrid local/global decoder layer:
 *
 *     O[b,h,t,:] = sum_s softmax_s( scale * <Q'[b,h,t,:], K'[b,g(h),s,:]> + M[t,s] ) V[b,g(h),s,:]
 *
 * with g(h) = floor(h / (Hq/Hkv)) (consecutive query heads share one KV head), Q' and K'
 * the split-half RoPE rotations of Q and K, and M the causal or sliding-window mask.
 * Definitions, by page and section:
 *   "PLaMo 3アーキテクチャ徹底解析" (imoz.jp):
 *     §4.2 grouped-query attention;  §4.4 the cache stores K before RoPE, positions are
 *     generated inside attention (keys 0..S-1, queries S-T..S-1), the local cache keeps
 *     the last W-1 tokens and re-numbers them;  §4.5 the attention equation, scale
 *     1/sqrt(d), no softcap;  §5.1 the masks (causal j <= i; window also i - j < W,
 *     self included);  §6.1 split-half RoPE, omega_j = theta^(-2j/d);  §6.3 YaRN
 *     frequencies and the amplitude factor on cos and sin;  §6.4 partial (p-)RoPE.
 *
 * Conventions (all entry points):
 *   - Tensors are bfloat16, dense, row-major in the layouts stated per call, in device
 *     memory, 16-byte aligned.  The caller owns every buffer, descriptor array, workspace
 *     and stream; the library allocates nothing.  Its only device state is a status word
 *     per GPU and the fixed 16 MiB scratch array of gqa_attn_decode_static, both
 *     compiled into the library; on the host it remembers, per device, which kernels
 *     have had their shared-memory limit raised (a mutex guards that record, so calls
 *     may come from several host threads and may drive several GPUs in turn).
 *   - Every call validates its arguments on the host and returns a negative gqa_status
 *     without launching anything if they are wrong.  Otherwise it enqueues its kernels on
 *     `stream` (NULL = the legacy default stream) and returns GQA_OK without waiting.
 *   - Errors found on the device (a bounded wait that expired, a full cache, an index
 *     out of range) are recorded in the device status word and returned by the next
 *     gqa_get_device_status().  Device code never traps.
 *   - Stream order holds as for any kernel.  On a stream that is not being captured,
 *     gqa_kv_append and the decode calls launch with programmatic stream serialization
 *     and let the next kernel begin launching early.  Each of their kernels waits for its
 *     predecessor before reading.  A caller's own kernel launched after them with that
 *     attribute must likewise execute griddepcontrol.wait (cudaGridDependencySynchronize)
 *     before it reads their outputs.
 *   - Head dims: prefill and decode d in {128, 256, 512}; kv_append, rope_apply and the
 *     Q/K normalisation d in {64, 128, 256, 512}.  Query group G = Hq/Hkv must be an
 *     integer; decode needs G <= 8.  Other values return GQA_ERR_UNSUPPORTED.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *gqa_stream_t;

typedef enum gqa_status {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = -1,     /* null pointer, non-positive size, inconsistent shape */
    GQA_ERR_UNSUPPORTED = -2,     /* head dim / group size / device not supported */
    GQA_ERR_ALIGNMENT = -3,       /* a pointer is not 16-byte aligned */
    GQA_ERR_CAPACITY = -4,        /* a linear cache is full, or a length exceeds a bound */
    GQA_ERR_CUDA = -5,            /* a CUDA runtime call failed */
    GQA_ERR_DEVICE_TIMEOUT = -6,  /* a device-side bounded wait expired */
    GQA_ERR_WORKSPACE = -7,       /* workspace missing or too small */
    GQA_ERR_RANGE = -8,           /* a position lies beyond the RoPE table */
    GQA_ERR_DEVICE_BOUNDS = -9    /* debug build only: a device-side index check failed */
} gqa_status;

/* ---- RoPE frequencies and table ---------------------------------------------------
 * gqa_rope_inv_freq (host only, no GPU needed): writes omega_j, j = 0..d/2-1, to out:
 *   omega_j = base^(-2j/d)                                        ("PLaMo 3..." §6.1)
 *   if yarn_factor != 1 (YaRN, §6.3):
 *     j_low  = (d/2) ln(yarn_L0 / (2 pi beta_fast)) / ln(base)   (not rounded)
 *     j_high = (d/2) ln(yarn_L0 / (2 pi beta_slow)) / ln(base)
 *     alpha_j = clip((j - j_low) / (j_high - j_low), 0, 1)
 *     omega_j *= (1 - alpha_j) + alpha_j / yarn_factor
 *   if rotate_fraction < 1 (p-RoPE, §6.4): omega_j = 0 for j >= round(rotate_fraction d/2);
 *     the exponent keeps the full d.
 * Returns GQA_ERR_INVALID_ARG for d odd/<= 0, base <= 1, yarn_factor < 1, or a fraction
 * outside (0, 1]. */
gqa_status gqa_rope_inv_freq(double *out, int d, double base, double yarn_factor,
                             double yarn_L0, double beta_fast, double beta_slow,
                             double rotate_fraction);

/* YaRN amplitude 1 + 0.1 ln(s) applied to both cos and sin (§6.3); host only. */
double gqa_yarn_amplitude(double s);

/* Bytes of a RoPE table for head dim d and positions 0..max_pos-1:
 * max_pos * (d/2) * 2 floats. */
size_t gqa_rope_table_bytes(int d, int max_pos);

/* Fills `table` (device, caller-owned, gqa_rope_table_bytes(d, max_pos) bytes) with
 * float pairs table[p*(d/2) + j] = (amp cos(p omega_j), amp sin(p omega_j)) for
 * p < max_pos: the angle and both functions are evaluated in double precision on the
 * device and rounded once to float.  inv_freq: host array of d/2 doubles (see above),
 * copied into the launch, so it may be freed on return.  d <= 512, amp > 0. */
gqa_status gqa_rope_table_build(float *table, const double *inv_freq, int d, double amp,
                                int max_pos, gqa_stream_t stream);

/* ---- RoPE application (§6.1) --------------------------------------------------------
 * y[b,h,t,:] = rotation of x[b,h,t,:] at position pos0 + t, pairs (j, j+d/2), using the
 * table (table_len positions).  x, y: [B, H, T, d] bf16; y may equal x (in place).
 * Each output is rounded once to bf16 from the float rotation. */
gqa_status gqa_rope_apply(const void *x, void *y, int B, int H, int T, int d, int pos0,
                          const float *table, int table_len, gqa_stream_t stream);

/* ---- Prefill (§4.4, §4.5, §5.1) ------------------------------------------------------
 * q: [B, Hq, T, d], k, v: [B, Hkv, S, d] (k before RoPE, as a cache holds it),
 * o: [B, Hq, T, d] bf16.  lse: [B, Hq, T] float32 natural-log sum of exp of the scaled
 * scores, or NULL.  T <= S; query t sits at position S - T + t, key s at position s.
 * window <= 0: full causal; window > 0: keys with q_pos - k_pos < window (self included).
 * scale multiplies the dot products (e.g. 1/sqrt(d)); the table's amplitude multiplies
 * them by amp^2 on top.  scale must be finite and > 0 (the softmax takes each row's
 * maximum before scaling), else GQA_ERR_INVALID_ARG.  table_len >= S.
 * Key tiles wholly outside [q_pos - window + 1, q_pos] are never loaded or multiplied.
 * k_is_rotated = 0: k holds keys before RoPE (as the PLaMo cache stores them, §4.4); they
 *   are rotated once at positions 0..S-1 into `workspace`, which must hold at least
 *   gqa_prefill_workspace_bytes(B, Hkv, S, d) bytes; its contents are undefined afterwards.
 * k_is_rotated = 1: k already carries RoPE (a cache that stores rotated keys, as Gemma's
 *   does, §4.4); workspace may be NULL.
 * k_is_rotated = 2 (d = 128 only, else GQA_ERR_UNSUPPORTED): k holds keys before RoPE and
 *   each K tile is rotated in shared memory as it lands, inside the attention kernel (RoPE
 *   fused into the tile load); workspace may be NULL.  Same results as 0, bit for bit.
 *   Slower than 0 on long inputs: a K tile is rotated again every time a query block
 *   reloads it, while 0 rotates each key once.  Any other value: GQA_ERR_INVALID_ARG.
 * Supports d = 128, 256, 512.  Hq % Hkv == 0. */
size_t gqa_prefill_workspace_bytes(int B, int Hkv, int S, int d);
gqa_status gqa_attn_prefill(const void *q, const void *k, const void *v, void *o,
                            float *lse, int B, int T, int S, int Hq, int Hkv, int d,
                            int window, float scale, const float *table, int table_len,
                            int k_is_rotated, void *workspace, size_t workspace_bytes,
                            gqa_stream_t stream);

/* ---- KV cache (§4.4) -----------------------------------------------------------------
 * One descriptor per sequence, in device memory, owned by the caller.
 *   k, v   : device [Hkv, cap, d] bf16, K stored before RoPE.
 *   rope   : device RoPE table for this sequence's layer type; rope_len positions.
 *            Decode at d = 512 treats a group of 32 pairs whose rows 0 and 1 are all
 *            exactly (1, 0) as never rotating (omega = 0 at amplitude 1, as
 *            gqa_rope_table_build writes p-RoPE's unrotated pairs) and reads no further
 *            rows of it.
 *   cap    : slots per KV head.
 *   count  : linear cache (is_ring = 0): tokens held; they occupy slots 0..count-1 and
 *            sit at positions equal to their slots.
 *            ring cache (is_ring = 1, cap = window W): tokens appended so far; token i
 *            lives in slot i mod cap.  Attention sees the newest min(count, cap) tokens,
 *            re-numbered 0..R-1 from oldest to newest (the last W-1 kept plus the new one).
 */
typedef struct gqa_kv_desc {
    void *k;
    void *v;
    const float *rope;
    int32_t cap;
    int32_t count;
    int32_t is_ring;
    int32_t rope_len;
} gqa_kv_desc;

/* Appends one token per sequence: k_new, v_new [nseq, Hkv, d] bf16 are written to slot
 * count (linear) or count mod cap (ring) of every KV head, then count += 1.  slots_out
 * (device int32[nseq], nullable) receives the slot written.  A full linear cache is not
 * written; its slot_out is -1 and the status word records GQA_ERR_CAPACITY. */
gqa_status gqa_kv_append(gqa_kv_desc *descs, int nseq, const void *k_new,
                         const void *v_new, int Hkv, int d, int32_t *slots_out,
                         gqa_stream_t stream);

/* ---- Chunked prefill over a cache (§4.4) ----------------------------------------------
 * A chunk of T new tokens of one sequence attends to the R tokens its cache holds
 * (linear: R = count; ring: R = min(count, cap), the newest ones, oldest first) followed
 * by itself: S = R + T keys at positions 0..S-1 and queries at R..S-1 (a local layer's
 * ring is re-numbered from 0, §4.4; its window W = cap covers every key a chunk query can
 * see).  Per chunk: gqa_prefill_gather, then gqa_attn_prefill(q [1, Hq, T, d], k_out,
 * v_out, B = 1, T, S, ..., k_is_rotated = 1), then gqa_kv_append_chunk.
 *
 * gqa_prefill_gather: desc is one device descriptor; k_new, v_new [Hkv, T, d] are the
 * chunk's keys (before RoPE) and values; k_out, v_out [Hkv, S, d] (caller-owned) receive
 * the S keys rotated at positions 0..S-1 and the S values.  S is the caller's count of
 * R + T; if the descriptor disagrees, or S > table_len, nothing is written and the status
 * word records GQA_ERR_CAPACITY (resp. GQA_ERR_RANGE).
 *
 * gqa_kv_append_chunk: k_new, v_new [nseq, Hkv, T, d]; each sequence's T tokens go to slots
 * count .. count + T - 1 (linear; if they do not fit, nothing is written and the status
 * word records GQA_ERR_CAPACITY) or (count + t) mod cap (ring; when T > cap only the last
 * cap tokens are stored), then count += T.  d in {64, 128, 256, 512}. */
gqa_status gqa_prefill_gather(const gqa_kv_desc *desc, const void *k_new, const void *v_new,
                              int T, int Hkv, int d, void *k_out, void *v_out, int S,
                              const float *table, int table_len, gqa_stream_t stream);
gqa_status gqa_kv_append_chunk(gqa_kv_desc *descs, int nseq, const void *k_new,
                               const void *v_new, int T, int Hkv, int d, gqa_stream_t stream);

/* ---- Q/K normalisation in front of attention (§3.2, §4.3, §4.4) ----------------------
 * RMSNorm with an effective gain (§3.2): N(x) = gamma * x / sqrt(mean(x^2) + eps) over
 * each (token, head) vector of d values; PLaMo's q_norm / k_norm use offset 1, so the
 * caller passes gamma = 1 + w (the stored weight w plus the offset), eps = 1e-6, and one
 * gain of d floats shared by every head (§4.3).  The order is fixed by §4.4: normalise,
 * store K in the cache (normalised, not rotated), then rotate.  Sums of squares and the
 * scaling run in fp32; each output is rounded once to bf16 (the public implementation's
 * intermediate bf16 rounding is not reproduced).  d in {64, 128, 256, 512}; gains are
 * device fp32 [d], 16-byte aligned; outputs may alias their inputs (q_out == q, k_out == k).
 *
 * Prefill form: q [B, Hq, T, d] -> q_out = N_q(q) (rotated later, inside
 * gqa_attn_prefill); k [B, Hkv, T, d] -> k_out = N_k(k) (what the cache stores, nullable)
 * and k_rot = RoPE(N_k(k)) at positions pos0 + t (nullable; pass it to gqa_attn_prefill
 * with k_is_rotated = 1).  V is not touched.  table as for gqa_rope_apply; positions
 * past table_len return GQA_ERR_RANGE. */
gqa_status gqa_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out, void *k_rot,
                            int B, int Hq, int Hkv, int T, int d, int pos0,
                            const float *q_gamma, const float *k_gamma, float eps,
                            const float *table, int table_len, gqa_stream_t stream);

/* Decode form: for each sequence one new token.  q [nseq, Hq, d] -> q_out = N_q(q) (the
 * decode kernel rotates it); k_new [nseq, Hkv, d] -> N_k(k_new) and v_new [nseq, Hkv, d]
 * (unchanged, or with v_norm = 1 normalised without a gain, as Gemma 4 does) are appended
 * to each sequence's cache exactly as gqa_kv_append appends them (slot, count update,
 * slots_out, GQA_ERR_CAPACITY on a full linear cache). */
gqa_status gqa_qk_norm_append(gqa_kv_desc *descs, int nseq, const void *q, const void *k_new,
                              const void *v_new, int Hq, int Hkv, int d, const float *q_gamma,
                              const float *k_gamma, float eps, int v_norm, void *q_out,
                              int32_t *slots_out, gqa_stream_t stream);

/* ---- Shared K/V projection (Gemma 4 global layers) ---------------------------------------
 * attention_k_eq_v ("PLaMo 3..." §5.2 and the Gemma 4 comparison of §8): one projection
 * output Z [.., Hkv, .., d] per token gives both K = RoPE(N_{gamma_k}(Z)) and V = N_1(Z),
 * N_1 being RMSNorm without a gain (eps as above).  Such a layer needs to cache only
 * Zn = N_1(Z): since N_gamma(Z) = gamma * N_1(Z), the keys are recomputed from it.  The
 * library does exactly that: the stored row is Zn rounded once to bf16, and the key is
 * RoPE(gamma_k * Zn) -- the fp32 gain times the stored row, rotated in fp32 and rounded
 * once to bf16 -- in prefill and decode alike (the two may round the rotation's products
 * in a different order, at most one bf16 step apart).  Gains are device fp32
 * [d], 16-byte aligned, one per layer, shared by every head; d in {64, 128, 256, 512}
 * (decode: {128, 256, 512}).
 *
 * gqa_qk_norm_rope_kv_shared (prefill form): q [B, Hq, T, d] -> q_out = N_{q_gamma}(q)
 * (rotated later, inside gqa_attn_prefill); z [B, Hkv, T, d] -> v_out = Zn (the values,
 * and what the cache stores; nullable) and k_rot = RoPE(gamma_k * Zn) at positions
 * pos0 + t (nullable; pass it to gqa_attn_prefill with k_is_rotated = 1 and v_out as v).
 * q, q_out and q_gamma may all be NULL (then Hq is ignored) to process Z alone; at least
 * one of v_out, k_rot must be given; k_gamma and the table are needed only for k_rot.
 * Each output may alias its own input (q_out == q; v_out or k_rot == z), not another output.
 *
 * gqa_kv_shared_append (decode form): q [nseq, Hq, d] -> q_out = N_{q_gamma}(q);
 * z_new [nseq, Hkv, d] -> Zn appended to each sequence's cache at desc.k, with the slot,
 * count update, slots_out and GQA_ERR_CAPACITY of gqa_kv_append; desc.v is not written.
 *
 * gqa_attn_decode_kv_shared: as gqa_attn_decode (same arguments, workspace and results),
 * over caches of Zn at desc.k: keys RoPE(k_gamma * Zn) at positions 0..R-1, values
 * Zn; desc.v is not read.  The cache rows are read once from memory for both roles, half
 * the bytes of separate K and V caches. */
gqa_status gqa_qk_norm_rope_kv_shared(const void *q, const void *z, void *q_out, void *v_out,
                                      void *k_rot, int B, int Hq, int Hkv, int T, int d,
                                      int pos0, const float *q_gamma, const float *k_gamma,
                                      float eps, const float *table, int table_len,
                                      gqa_stream_t stream);
gqa_status gqa_kv_shared_append(gqa_kv_desc *descs, int nseq, const void *q, const void *z_new,
                                int Hq, int Hkv, int d, const float *q_gamma, float eps,
                                void *q_out, int32_t *slots_out, gqa_stream_t stream);

/* ---- Decode (§4.4, §4.5) ---------------------------------------------------------------
 * One query token per sequence: q [nseq, Hq, d] bf16 at position R-1, where R = count
 * (linear) or min(count, cap) (ring) read from the descriptors (so call after
 * gqa_kv_append).  Keys are the R logical tokens at positions 0..R-1, rotated on the fly
 * with the sequence's table.  o: [nseq, Hq, d] bf16; lse: [nseq, Hq] float or NULL.
 * max_len: an upper bound on R over the batch (sizes the split-KV grid); a sequence with
 * R > max_len or rope_len < R is skipped and flagged in the status word.
 * workspace: device scratch of gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len) bytes:
 * the split partials, nseq Hq nsplit (m, l) float pairs padded to a multiple of 4 floats,
 * then nseq Hq nsplit rows of d floats.  The number of splits per sequence, nsplit, and
 * the keys per split are chosen from (nseq, Hkv, d, max_len) so that the grid fills the
 * GPU; the workspace size follows the same rule, so it must be queried with the shape of
 * the call.  scale: finite and > 0.
 * d in {128, 256, 512} (Gemma-4 local / global heads), Hq/Hkv <= 8. */
size_t gqa_decode_workspace_bytes(int nseq, int Hq, int Hkv, int d, int max_len);
gqa_status gqa_attn_decode(const void *q, const gqa_kv_desc *descs, int nseq, int Hq,
                           int Hkv, int d, float scale, int max_len, void *o, float *lse,
                           void *workspace, size_t workspace_bytes, gqa_stream_t stream);

gqa_status gqa_attn_decode_kv_shared(const void *q, const gqa_kv_desc *descs, int nseq, int Hq,
                                     int Hkv, int d, float scale, const float *k_gamma,
                                     int max_len, void *o, float *lse, void *workspace,
                                     size_t workspace_bytes, gqa_stream_t stream);

/* Decode without a caller-supplied workspace; allocates nothing.  The pages have no
 * counterpart to this entry point: it is the same computation as gqa_attn_decode (same
 * kernels, same arguments and results), for callers that cannot provide scratch memory --
 * for instance because their device memory is owned by another component (a framework
 * allocator that reserved the GPU up front, a serving loop that forbids allocation), or
 * because the device synchronisation of cudaMalloc/cudaFree is unacceptable per step.
 * The split-KV partials go to a fixed 16 MiB device array inside the library, which every
 * GPU that loads the library holds until the process exits.  A call whose partials need
 * more than that, i.e. gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len) > 16 MiB, returns
 * GQA_ERR_WORKSPACE without launching.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture.
 * All calls share the one array and it keeps the last call's contents (each call writes
 * every record it reads, so no clearing is needed): calls that may overlap on the GPU --
 * on different streams, or from different host threads -- race on it and must be
 * serialised by the caller. */
gqa_status gqa_attn_decode_static(const void *q, const gqa_kv_desc *descs, int nseq, int Hq,
                                  int Hkv, int d, float scale, int max_len, void *o,
                                  float *lse, gqa_stream_t stream);

/* ---- Status ----------------------------------------------------------------------------
 * Waits for `stream`, then returns and clears the current device's status word
 * (GQA_OK if no device-side error was recorded since the last call). */
gqa_status gqa_get_device_status(gqa_stream_t stream);

/* Waits for `stream`, then stores in diag[0..n) and clears the diagnostic codes of the
 * device-side bounded waits that expired since the last call (0 where none): diag[0] the
 * first overall, diag[1..4] the first of each kernel role 0..3.  A code is
 * (kernel << 24) | (role << 20) | (barrier << 16) | (tile index & 0xffff), kernel 1 =
 * prefill d=128, 2 = prefill d=256, 3 = decode, 4 = gqa_watchdog_selftest,
 * 5 = prefill d=512 (a pair of CTAs), 6 = cache append, chunk gather, RoPE pass, Q/K
 * normalisation.  A library compiled with -DGQA_DEBUG_BOUNDS checks the indices of the
 * global accesses it derives from device-side data; the first failed check records
 * GQA_ERR_DEVICE_BOUNDS and, in diag[0], (kernel << 24) | (1 << 23) | site, and the access
 * is skipped.  For diagnosing device-side errors; gqa_get_device_status leaves the codes
 * in place. */
gqa_status gqa_get_device_diag(gqa_stream_t stream, int32_t *diag, int n);

/* Self-test of the device-side watchdog (the pages have no counterpart: this checks the
 * library's own failure detection).  Enqueues on `stream` one warp that waits on an
 * mbarrier nothing ever arrives on, bounded by limit_ns nanoseconds, with the same wait
 * and reporting code as the attention kernels.  The wait expires, the kernel records
 * GQA_ERR_DEVICE_TIMEOUT and diagnostic code 4 << 24 and returns normally: the next
 * gqa_get_device_status returns GQA_ERR_DEVICE_TIMEOUT and the context stays usable.
 * limit_ns in [1000, 2000000000] (1 us .. 2 s, the kernels' own limit), else
 * GQA_ERR_INVALID_ARG without launching. */
gqa_status gqa_watchdog_selftest(int64_t limit_ns, gqa_stream_t stream);

/* Static, human-readable text for a status code. */
const char *gqa_status_string(int status);

/* Text of the CUDA runtime error behind the most recent GQA_ERR_CUDA returned to the
 * calling host thread (static storage; "no CUDA error recorded" if there was none). */
const char *gqa_last_error_string(void);

/* GQA_OK if the current CUDA device is an sm_103 part this build can run on. */
gqa_status gqa_device_check(void);

#ifdef __cplusplus
}
#endif
#endif /* GQA_ATTN_H */
