/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated-delta-rule library, libgdn.so.
 *
 * The operation (one call = a whole run of steps for every sequence and head):
 *
 *   for each sequence b and head h, starting from S = state_in[b,h]:
 *     for t = 0 .. n_tokens-1:
 *       S   = exp(g[b,t,h]) * S * (I - beta[b,t,h] k k^T) + beta[b,t,h] v k^T
 *       out[b,t,h,:] = S q / sqrt(head_dim)
 *     state_out[b,h] = S
 *   with q, k, v the vectors q[b,t,h,:], k[b,t,h,:], v[b,t,h,:].
 *
 * Sources:
 *   - "marcsun13/ggml-gated-delta-net" model card, section "Ops": the op is
 *     one dispatch for a whole run of gated-delta-rule steps with signature
 *     (q, k, v, g, beta, state) -> (out, final_state); the shape table
 *     (q, k, v: (n_seqs, n_tokens, n_heads, head_dim); g, beta: (n_seqs,
 *     n_tokens, n_heads); state: (n_seqs, n_heads, head_dim, head_dim));
 *     the contract notes under it: one key head per value head (identity
 *     mapping), state indexed [value][key] and returned in the same layout,
 *     a fresh state is zeros, the output carries 1/sqrt(head_dim), g is a
 *     log-domain gate that the kernel exponentiates, and the head_dim
 *     capability query.
 *   - "marcsun13/ggml-gated-delta-net" model card, section "Where the kernels
 *     come from": work is enqueued on the caller's queue, never as a
 *     separate submission.  Here: every call only enqueues on `stream`.
 *   - "Gated Delta Net on AMD: why ROCm stumbles on hybrid-attention LLMs",
 *     section "What Gated Delta Net is, in plain language": delta rule
 *     (overwrite what new information contradicts) plus a gate (how much
 *     of the old state is kept).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, dense and
 *     row-major in the torch order above.  q, k, v, out, state_in and
 *     state_out must be 16-byte aligned; g and beta 4-byte aligned.
 *   - g and beta are float32.  state_in / state_out are float32 [value][key].
 *     out is float32 (n_seqs, n_tokens, n_heads, head_dim), already scaled
 *     (bfloat16 with the GDN_OPT_OUT_BF16 option of gdn_forward_ex).
 *   - state_in may be NULL: the initial state is then zeros.
 *   - state_out == state_in (the same pointer) updates the state in place.
 *     Any other overlap between an output (out, state_out) and any other
 *     buffer is rejected with GDN_ERR_ALIAS.
 *   - q and k are used as given: the op does not L2-normalise them (the
 *     GDN_OPT_L2NORM_QK option of gdn_forward_ex does).
 *   - Sizes: n_seqs, n_heads >= 0, n_tokens >= 0.  A call with n_seqs == 0 or
 *     n_heads == 0 does nothing.  n_tokens == 0 copies state_in (or zeros)
 *     into state_out and writes no output.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and never synchronise the host.
 *   - Return value: GDN_OK (0), or a negative GDN_ERR_* code.  Argument
 *     errors are detected on the host before anything is enqueued: nothing
 *     is launched and nothing is written.  GDN_ERR_CUDA reports a failed
 *     launch or enqueue (the CUDA error is then available from
 *     cudaGetLastError-like queries by the caller).  Faults that happen
 *     later on the device are reported by gdn_get_device_status().
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t. */
typedef struct CUstream_st *gdn_stream_t;

enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_ARG = -1,       /* NULL pointer for a non-empty tensor, negative size, size overflow */
    GDN_ERR_HEADDIM = -2,   /* head_dim not supported on the requested path (see gdn_supports) */
    GDN_ERR_ALIGN = -3,     /* pointer misaligned (16 B for tensors, 4 B for g/beta) */
    GDN_ERR_ALIAS = -4,     /* an output overlaps an input or the other output */
    GDN_ERR_CUDA = -5,      /* a CUDA launch / enqueue / allocation call failed */
    GDN_ERR_TIMEOUT = -6,   /* a bounded device-side wait gave up (gdn_get_device_status) */
    GDN_ERR_WORKSPACE = -7, /* caller workspace NULL, too small or misaligned */
    GDN_ERR_NOMEM = -8,     /* stream-ordered workspace allocation failed */
    GDN_ERR_DTYPE = -9,     /* dtype not supported on the requested path (chunked: bf16 only) */
    GDN_ERR_SHAPE = -10,    /* shape outside the op's scope (flash_attn: 20 or more queries) */
    GDN_ERR_SCRATCH = -11   /* gdn_forward_noalloc: the call needs more than its fixed scratch */
};

/* dtype of q, k, v (F16: decode attention only) */
enum gdn_dtype { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1, GDN_DTYPE_F16 = 2 };

/* execution path; AUTO picks by n_tokens and head_dim */
enum gdn_path { GDN_PATH_AUTO = 0, GDN_PATH_RECURRENT = 1, GDN_PATH_CHUNKED = 2 };

/*
 * Options, OR-ed into the `path` argument of gdn_forward_ex,
 * gdn_forward_noalloc and gdn_workspace_bytes (bits above the low byte;
 * unknown bits are rejected with GDN_ERR_ARG).
 *
 * GDN_OPT_L2NORM_QK: q and k are L2-normalised inside the op, per (sequence,
 *   token, key head) over head_dim: x -> x / |x|, in float32, a zero vector
 *   staying zero (a vector whose squared norm underflows float32 counts as
 *   zero).  The call then computes the recurrence of the normalised q and k.
 *   This is one of the eager operations that the model card ("Ops") counts
 *   around the recurrence of a Gated DeltaNet layer; fused here it saves a
 *   read and a write of q and k.  Both paths and every head_dim serve it; on
 *   the chunked path the norms are applied as per-token scalars in float32,
 *   so raw bf16 q and k still enter the tensor-core products exactly.
 */
#define GDN_OPT_L2NORM_QK 0x100

/*
 * GDN_OPT_OUT_BF16: `out` is bfloat16 (raw 16-bit words, __nv_bfloat16
 *   layout), same shape, still scaled by 1/sqrt(head_dim).  Each element is
 *   the float32 value the call writes without this option, rounded to
 *   nearest even; the recurrence and the state stay float32.  The call then
 *   needs half the output bytes (its size, alignment and overlap checks count
 *   2-byte elements).  The extra error is that one rounding: at most 2^-8 of
 *   each element's magnitude (bf16 keeps an 8-bit significand).
 */
#define GDN_OPT_OUT_BF16 0x200

/*
 * gdn_forward -- the op with float32 q, k, v.
 * q, k, v: (n_seqs, n_tokens, n_heads, head_dim) float32.  Other arguments as
 * described above.  Uses the AUTO path; if that path needs a workspace it is
 * allocated and released in stream order on `stream` (no host
 * synchronisation) from a memory pool the library keeps per device, which
 * holds up to 1 GiB reserved between calls.
 */
int gdn_forward(const float *q, const float *k, const float *v,
                const float *g, const float *beta, const float *state_in,
                float *out, float *state_out,
                int n_seqs, int n_tokens, int n_heads, int head_dim,
                gdn_stream_t stream);

/* gdn_forward_bf16 -- as gdn_forward with bfloat16 q, k, v (raw 16-bit
 * words, __nv_bfloat16 layout).  Computation is float32 with exact upcast. */
int gdn_forward_bf16(const void *q, const void *k, const void *v,
                     const float *g, const float *beta, const float *state_in,
                     float *out, float *state_out,
                     int n_seqs, int n_tokens, int n_heads, int head_dim,
                     gdn_stream_t stream);

/*
 * gdn_forward_ex -- explicit key-head count, dtype, path and workspace.
 * n_k_heads: number of heads q and k carry; 0 means n_heads.  q and k are
 *   then (n_seqs, n_tokens, n_k_heads, head_dim) and value head i reads key
 *   (and query) head i % n_k_heads -- the tiled mapping that the model card's
 *   contract notes under the "Ops" shape table give for upstream; with
 *   n_k_heads == n_heads it is the identity.  n_k_heads must divide n_heads
 *   (else GDN_ERR_ARG).  v, g, beta, out and the state keep n_heads heads.
 * dtype: GDN_DTYPE_*; path: GDN_PATH_*, optionally OR-ed with GDN_OPT_* flags.
 * workspace: caller-owned device buffer of at least
 *   gdn_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, dtype, path)
 *   bytes, 256-byte aligned; or NULL, in which case the call allocates and
 *   frees it stream-ordered on `stream` from the library's per-device memory
 *   pool (cudaMallocFromPoolAsync / cudaFreeAsync; up to 1 GiB stays
 *   reserved in the pool between calls).
 * The workspace contents on entry are ignored; on return they are garbage.
 * Two calls in flight at once must not share a workspace.
 */
int gdn_forward_ex(const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const float *state_in,
                   float *out, float *state_out,
                   int n_seqs, int n_tokens, int n_heads, int n_k_heads, int head_dim,
                   int dtype, int path, void *workspace, size_t workspace_bytes,
                   gdn_stream_t stream);

/*
 * gdn_forward_noalloc -- gdn_forward_ex for callers that cannot allocate
 * device memory while they run (for example a serving framework that has
 * reserved the whole device for its own arena, or a decode loop that must
 * not stall on an allocation).  This entry point has no counterpart in the
 * paper or the model card; it exists only for such callers.
 *
 * Same arguments and behaviour as gdn_forward_ex, without the workspace
 * arguments.  It calls no allocation routine.  The chunked calls that need
 * scratch (head_dim 256, and head_dim 128 with fewer than 80 (sequence, head)
 * pairs: 32 KiB per sequence, head and 64-token chunk) use a fixed array of
 * GDN_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library, held by every GPU
 * that loads the library until the process exits.
 * A call that would need more returns GDN_ERR_SCRATCH before touching the
 * GPU; gdn_workspace_bytes() tells how much a call needs.
 * All calls share the array: calls that may overlap on the GPU (different
 * streams with no ordering) race on it and must not be issued that way.  Its
 * contents carry over between calls; no call depends on them.
 * The first call on each device that needs the array looks up its device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
int gdn_forward_noalloc(const void *q, const void *k, const void *v,
                        const float *g, const float *beta, const float *state_in,
                        float *out, float *state_out,
                        int n_seqs, int n_tokens, int n_heads, int n_k_heads, int head_dim,
                        int dtype, int path, gdn_stream_t stream);

/* Bytes of device workspace gdn_forward_ex needs for these sizes, dtype and
 * path (0 when the selected path needs none).  Only chunked calls need one:
 * head_dim 256, and head_dim 128 with fewer than 80 (sequence, head) pairs,
 * which run a chunk-transform kernel and a state kernel; 32 KiB per
 * sequence, head and 64-token chunk.  Returns 0 on invalid sizes. */
size_t gdn_workspace_bytes(int n_seqs, int n_tokens, int n_heads, int head_dim,
                           int dtype, int path);

/* Which path AUTO selects (GDN_PATH_RECURRENT or GDN_PATH_CHUNKED) for
 * these sizes and dtype, or a negative GDN_ERR_* for unsupported ones.
 * AUTO takes the chunked path for bf16 q/k/v, head_dim 64/128/256 and at
 * least T_switch tokens, everything else runs the recurrent path.  T_switch
 * was measured on GB300 and depends on head_dim and on the number of
 * (sequence, head) pairs P = n_seqs * n_heads:
 *   head_dim 64: 48 (P < 1024) or 64;  128: 72 (P < 48), 44 (P < 80) or 24;
 *   256: 32 (P < 128) or 24. */
int gdn_select_path(int n_seqs, int n_tokens, int n_heads, int head_dim, int dtype);

/*
 * gdn_supports -- capability query, the counterpart of the model card's
 * supports_gated_delta_net(head_dim) ("Ops" table and the note that the
 * head dim must be asked, not assumed).  Returns a bit mask: bit 0 (1) =
 * the recurrent path supports head_dim, bit 1 (2) = the chunked path does
 * (for bf16 q/k/v).  0 means unsupported.  Supported: 32 and 96 (recurrent
 * only), 64, 128, 256 (both).  The model card's shape note says upstream
 * covers a state row with 32 threads, so its head_dim is a multiple of 32 up
 * to 128; every such width is served here, and 256 as well.
 */
int gdn_supports(int head_dim);

/*
 * gdn_get_device_status -- synchronises `stream`, then returns and clears
 * the library's device status word on the current device: GDN_OK, or
 * GDN_ERR_TIMEOUT if a kernel's bounded wait gave up since the last query.
 * Returns GDN_ERR_CUDA if the synchronisation itself failed.
 */
int gdn_get_device_status(gdn_stream_t stream);

/*
 * gdn_flash_attn -- decode attention, the flash_attn op of the model card
 * ("marcsun13/ggml-gated-delta-net", section "flash_attn": shape table, the
 * vector variant for fewer than 20 queries, grouped-query attention with k
 * and v passed unexpanded, additive mask, result with tokens before heads):
 *
 *   out[b, i, h, :] = sum_j softmax_j(scale * q[b,h,i,:] . k[b,hk,j,:]
 *                                     + mask[b,0,i,j]) * v[b,hk,j,:]
 *   hk = h / (n_heads / n_heads_kv)          (grouped heads, as repeat_kv)
 *
 * q:    (n_seqs, n_heads, n_q, head_dim_k)        dtype
 * k:    (n_seqs, n_heads_kv, n_kv, head_dim_k)    dtype
 * v:    (n_seqs, n_heads_kv, n_kv, head_dim_v)    dtype
 * mask: (n_seqs, 1, n_q, n_kv) dtype, additive (-inf masks a key), or NULL
 * out:  (n_seqs, n_q, n_heads, head_dim_v) float32, written by the call
 * dtype: GDN_DTYPE_F32, GDN_DTYPE_BF16 or GDN_DTYPE_F16 for q, k, v and the
 *   mask together; accumulation is float32 and q, k, v enter exactly (for
 *   16-bit inputs through tensor-core MMAs, the softmax weights as hi + lo
 *   16-bit pairs, about 16 significant bits).
 * scale: finite float multiplying q . k (callers usually pass
 *   1 / sqrt(head_dim_k)).
 * Supported: 1 <= n_q <= 19 (else GDN_ERR_SHAPE), head_dim_k and head_dim_v
 *   each in {64, 128, 256}, equal or not (the model card's capability query
 *   takes the two widths separately; else GDN_ERR_HEADDIM), n_heads_kv
 *   dividing n_heads (else
 *   GDN_ERR_ARG); any n_kv >= 0.  A query whose keys are all masked with
 *   -inf, and every query when n_kv == 0, gets a zero output row.
 * q, k, v, out 16-byte aligned; mask aligned to its element size; out must
 * not overlap an input (GDN_ERR_ALIAS).  Asynchronous on `stream`; argument
 * errors launch nothing.  Needs no workspace.
 */
int gdn_flash_attn(const void *q, const void *k, const void *v, const void *mask, float *out,
                   int n_seqs, int n_heads, int n_heads_kv, int n_q, int n_kv,
                   int head_dim_k, int head_dim_v, float scale, int dtype,
                   gdn_stream_t stream);

/* Capability query, the counterpart of supports_flash_attn(n_q, head_dim_k,
 * head_dim_v) in the model card's "Ops" table: 1 if gdn_flash_attn serves
 * that shape, 0 otherwise. */
int gdn_flash_attn_supports(int n_q, int head_dim_k, int head_dim_v);

/*
 * gdn_selftest_wait_timeout -- exercises the library's failure path on the
 * GPU without faulting it: enqueues on `stream` one small kernel whose
 * bounded wait (on a barrier nothing ever completes) gives up after about
 * 0.1 ms and records GDN_ERR_TIMEOUT in the device status word, the same way
 * the chunked kernels report a wait that gives up.  The kernel then returns
 * normally and the context stays usable; a following
 * gdn_get_device_status() returns GDN_ERR_TIMEOUT and clears it.  A
 * diagnostic with no counterpart in the pages.  Returns GDN_OK once enqueued.
 */
int gdn_selftest_wait_timeout(gdn_stream_t stream);

/* Static English text for a status code (never NULL). */
const char *gdn_status_string(int status);

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
