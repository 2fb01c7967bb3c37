/*
 * usp.h - C ABI of the GB300 sequence-parallel attention core.
 *
 * What the library computes
 * -------------------------
 * Exact softmax attention of every query shard against the KV shards of a
 * ring, in ring order, with the per-shard partials (O, LSE) merged by the
 * associative log-sum-exp rule so the result equals full attention
 * ("Long Context Attention" notes, sections "Ring Attention" and "Tree
 * Attention"; YunChang README, "2. Usage"; ring-sliding-window-attention
 * README, "Arguments"). cp_size ring ranks and ulysses_degree Ulysses ranks
 * are virtual: all of them live in one device's memory, the ring hop is an
 * address offset and the Ulysses all-to-all is a device-memory permute.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *    stated otherwise; the library never frees or retains it after the call
 *    returns, and allocates no device memory. Scratch space comes from a
 *    caller-provided workspace whose size the *_workspace_size calls give.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and never synchronises the host. Argument errors are detected
 *    on the host before anything is launched; the call then returns an error
 *    status and enqueues no work.
 *  - Tensor pointers must be 16-byte aligned (USP_ERR_ALIGNMENT otherwise).
 *  - Tensors are row-major with the layouts stated per call. "Permuted" or
 *    "rank-major" sequence order means the concatenation of ring rank 0's
 *    shard, rank 1's shard, ..., each shard in increasing natural position:
 *      contiguous: rank r holds positions [r*S/cp, (r+1)*S/cp)
 *      zigzag:     S is cut into 2*cp chunks of S/(2*cp); rank r holds chunk
 *                  r then chunk 2*cp-1-r ("Zig-Zag Attention": folding the
 *                  causal mask makes every cross-rank chunk pair a full
 *                  square or empty and balances the work)
 *      stripe:     rank r holds positions r, r+cp, r+2cp, ... ("Solution":
 *                  KV0 holds tokens 0,4,8,12 of 16 on 4 hosts)
 *  - With ulysses_degree ud > 1 the world is W = cp*ud ranks numbered
 *    w = rho*ud + u (rho = ring rank, u = Ulysses rank). Rank w's sequence
 *    shard is permuted positions [w*S/W, (w+1)*S/W).
 *
 * Masks. Query position i sees key position j (positions counted from the
 * start of their own sequence; keys of another packed sequence are never
 * visible) iff
 *     (!causal || j <= i) && (window <= 0 || i - j < window || j < sink_tokens)
 * `window` is the number of visible keys including the query itself
 * (ring-sliding-window README, "Arguments": window_size); `sink_tokens`
 * leading tokens of every sequence stay visible outside the window (the
 * README's "Ring Streaming LLM Attention"). A query that sees no key gets
 * O = 0 and LSE = -inf.
 */
#ifndef USP_H_
#define USP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *usp_stream_t;

typedef enum {
  USP_OK = 0,
  USP_ERR_INVALID_ARG = 1,  /* a size, degree, enum or pointer is invalid   */
  USP_ERR_UNSUPPORTED = 2,  /* valid, but this build has no kernel for it   */
  USP_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned             */
  USP_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required   */
  USP_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, attrs)   */
  USP_ERR_TIMEOUT = 6       /* a device wait gave up (reported by a kernel) */
} usp_status_t;

typedef enum {
  USP_LAYOUT_CONTIGUOUS = 0,
  USP_LAYOUT_ZIGZAG = 1,
  USP_LAYOUT_STRIPE = 2
} usp_layout_t;

typedef enum { USP_BF16 = 0, USP_FP32 = 1 } usp_dtype_t;

typedef enum {
  USP_PERMUTE_EXTRACT = 0,          /* natural order -> rank-major order  */
  USP_PERMUTE_RESTORE = 1,          /* rank-major order -> natural order  */
  USP_PERMUTE_ULYSSES_SEQ2HEAD = 2, /* Ulysses all-to-all before attention */
  USP_PERMUTE_ULYSSES_HEAD2SEQ = 3  /* Ulysses all-to-all after attention  */
} usp_permute_kind_t;

/* Flags for the attention calls. */
#define USP_FLAG_NONE 0u
/* Run the CUDA-core fp32 kernels even where the tensor-core kernels apply
 * (bf16 inputs). Used to cross-check the two kernel families. */
#define USP_FLAG_FORCE_SIMT 1u
/* usp_attn_bwd / usp_attn_bwd_qkvpacked with ulysses_degree > 1: reuse the
 * forward's Ulysses exchange instead of redoing it. The backward of the
 * method keeps the head-sharded q, k, v, output and LSE of the forward
 * ("Long Context Attention" notes, "Motivation": QKV, output, LSE and dout
 * are stored for the backward), so only dout goes through the sequence-to-
 * head exchange and dq, dk, dv through the way back. The caller passes the
 * backward the same workspace that the forward call with the same arguments
 * wrote (so it must be at least usp_attn_bwd_workspace_size bytes, which is
 * never less than the forward's size), untouched since: its first
 * usp_attn_fwd_workspace_size bytes then hold the forward's head-sharded
 * q, k, v and out, where the backward reads them. q, k, v, out are not read
 * and may be NULL. Ignored by the forward and when ulysses_degree == 1;
 * rejected (USP_ERR_INVALID_ARG) by usp_attn_bwd_noalloc. The contents of
 * the workspace are trusted: a workspace that does not hold that forward's
 * exchange gives wrong gradients, not an error. */
#define USP_FLAG_SAVED_EXCHANGE 2u
/* usp_attn_fwd / usp_attn_bwd (and usp_attn_bwd_noalloc): q, k, v, out,
 * dout, dq, dk and dv are in natural sequence order instead of rank-major
 * order; lse stays rank-major (it is the forward's state for the backward).
 * The result equals extracting the inputs (USP_PERMUTE_EXTRACT), calling
 * without the flag and restoring the outputs (USP_PERMUTE_RESTORE), bit for
 * bit (dq to rounding: its additions happen in hardware order). Where the
 * tensor-core kernels run, the layout is contiguous or zigzag (a 128-token
 * tile is then a run of natural positions) and the problem is short per
 * token (a window, a packed batch, or S <= 16384), they read and write the
 * caller's tensors in place, with no copy at all. Otherwise (longer dense
 * sequences, where copies cost less than reading in place; stripe; the
 * CUDA-core kernels) the extract and restore ride along with the Ulysses
 * exchange when ulysses_degree > 1, or run as copies into the workspace
 * when ulysses_degree == 1 (usp_attn_*_workspace_size must be given the
 * flag).
 * q, k, v, out must be passed to the backward even with
 * USP_FLAG_SAVED_EXCHANGE (which then only spares the copy path's copies).
 * Not supported by the q/k/v-packed entry points and usp_attn_fwd_fp8
 * (USP_ERR_UNSUPPORTED). Forward and backward must be given the same
 * flags. */
#define USP_FLAG_NATURAL_ORDER 4u

/*
 * usp_attn_fwd - ring attention forward with the fused LSE merge.
 *
 * Defines: per ring rank rho and step s = 0..cp-1, the partial attention of
 * rho's queries against the KV shard of rank (rho - s) mod cp ("Ring
 * Attention": KV segments circulate until every host has seen all of them),
 * merged in step order with the log-sum-exp rule ("Tree Attention":
 * logsumexp and max are associative). The merged running partial is kept
 * unnormalised (row max m, row sum l, sum of exp-weighted values) inside the
 * kernel; that representation is equivalent to (O = acc/l, LSE = m + log l).
 * With ulysses_degree > 1 (USP), q/k/v are first exchanged sequence->head
 * inside the workspace, each Ulysses group runs its ring over its H/ud
 * heads, and the output is exchanged head->sequence back into `out`.
 *
 * q    [B, S, Hq, D]   (packed: [S, Hq, D], S = total tokens T), rank-major
 *      (natural order with USP_FLAG_NATURAL_ORDER)
 * k, v [B, S, Hkv, D]  (packed: [S, Hkv, D]), same order and layout as q
 * out  [B, S, Hq, D]   written, in q's sequence order, dtype as q
 * lse  [B, Hq, S] fp32 written (packed: [Hq, S]), natural log of the scaled
 *      scores' sum of exponentials, rank-major sequence order
 * B, S, Hq, Hkv, D   D in {64, 128}; Hq % Hkv == 0 (query head h reads KV
 *      head h / (Hq/Hkv)); Hq % ud == 0 and Hkv % ud == 0 (Ulysses splits
 *      heads, YunChang README "Why not apply Ulysses ... individually");
 *      S % (cp*ud) == 0, zigzag also S % (2*cp*ud) == 0.
 * softmax_scale  <= 0 selects 1/sqrt(D) (the README's default).
 * causal, window, sink_tokens  the mask above. sink_tokens >= 0.
 * cu_seqlens  NULL for dense batches. Otherwise int32 [B + 1] device array
 *      of cumulative sequence lengths over the whole packed batch and all
 *      ranks (ring-sliding-window README, "Arguments": cu_seqlens is global,
 *      not per rank), cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] = S;
 *      B is then the number of sequences and the layout applies to the
 *      packed sequence. The values are trusted (not checked on the device):
 *      malformed boundaries give wrong masks but no out-of-bounds access.
 *      usp_check_cu_seqlens checks a host copy (the debug-mode check).
 * cp_size >= 1, ulysses_degree >= 1, layout, dtype (q/k/v/out element type).
 * flags  USP_FLAG_*.
 * workspace / workspace_bytes  caller scratch of at least
 *      usp_attn_fwd_workspace_size(...) bytes, 256-byte aligned (may be NULL
 *      when that size is 0). Its contents on entry are irrelevant. With
 *      ulysses_degree > 1 it holds the head-sharded q, k, v and out on
 *      return (what USP_FLAG_SAVED_EXCHANGE lets the backward reuse).
 * Errors: USP_ERR_INVALID_ARG, USP_ERR_ALIGNMENT, USP_ERR_WORKSPACE,
 *      USP_ERR_UNSUPPORTED (D not in {64,128}; USP_FLAG_NATURAL_ORDER from
 *      the packed entry point), USP_ERR_CUDA.
 */
usp_status_t usp_attn_fwd(const void *q, const void *k, const void *v,
                          void *out, float *lse, int B, int S, int Hq, int Hkv,
                          int D, float softmax_scale, int causal, int window,
                          int sink_tokens, const int32_t *cu_seqlens,
                          int cp_size, int ulysses_degree, usp_layout_t layout,
                          usp_dtype_t dtype, unsigned flags, void *workspace,
                          size_t workspace_bytes, usp_stream_t stream);

size_t usp_attn_fwd_workspace_size(int B, int S, int Hq, int Hkv, int D,
                                   int cp_size, int ulysses_degree,
                                   usp_dtype_t dtype, unsigned flags);

/*
 * usp_check_cu_seqlens - the debug-mode check of packed-sequence boundaries.
 *
 * The attention calls trust their cu_seqlens (a device array: checking it
 * would need a synchronisation). A caller that wants it checked copies it to
 * the host and passes the copy here (the boundaries of the packed batch, as
 * the ring-sliding-window README's "Arguments" define cu_seqlens: global over
 * all ranks): cu_seqlens_host [nseq + 1] int32, HOST
 * memory, read only. Returns USP_OK when cu_seqlens_host[0] == 0, the
 * values never decrease and cu_seqlens_host[nseq] == total_tokens (the S of
 * the attention call); else USP_ERR_INVALID_ARG, with the first offending
 * index in usp_last_error_detail(). nseq >= 1 and a non-NULL pointer are
 * required (USP_ERR_INVALID_ARG otherwise). Touches no device state.
 */
usp_status_t usp_check_cu_seqlens(const int32_t *cu_seqlens_host, int nseq, int total_tokens);

/*
 * usp_attn_bwd - gradients of usp_attn_fwd from the saved (out, lse).
 *
 * The LSE kept by the forward pass is what the backward pass needs ("Long
 * Context Attention" notes, "Motivation": QKV, output, LSE and dout are
 * stored for the backward). With P = exp(scale*q.k - LSE):
 *   Delta_i = <dO_i, O_i>, dV = P^T dO, dS = P * (dO V^T - Delta),
 *   dQ = scale dS K, dK = scale dS^T Q,
 * accumulated over every ring step; dK/dV of a shard collect the
 * contributions of every query rank that saw it (the shard's ring return)
 * and of all Hq/Hkv query heads sharing the KV head.
 *
 * q, k, v, out, lse: as passed to / produced by usp_attn_fwd (same args);
 *      with USP_FLAG_SAVED_EXCHANGE and ulysses_degree > 1, q, k, v, out are
 *      read from the forward's workspace instead (see the flag).
 * dout [B,S,Hq,D] in q's sequence order, dtype as q. dq/dk/dv written,
 *      shapes and order of q/k/v.
 * Scalar arguments must equal those of the forward call.
 * Errors: as usp_attn_fwd.
 */
usp_status_t usp_attn_bwd(const void *q, const void *k, const void *v,
                          const void *out, const float *lse, const void *dout,
                          void *dq, void *dk, void *dv, int B, int S, int Hq,
                          int Hkv, int D, float softmax_scale, int causal,
                          int window, int sink_tokens,
                          const int32_t *cu_seqlens, int cp_size,
                          int ulysses_degree, usp_layout_t layout,
                          usp_dtype_t dtype, unsigned flags, void *workspace,
                          size_t workspace_bytes, usp_stream_t stream);

size_t usp_attn_bwd_workspace_size(int B, int S, int Hq, int Hkv, int D,
                                   int cp_size, int ulysses_degree,
                                   usp_dtype_t dtype, unsigned flags);

/*
 * usp_attn_bwd_noalloc - usp_attn_bwd for callers that cannot allocate.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot provide a workspace: a runtime that has already handed all device
 * memory to its own pools, or code on a path where cudaMalloc is not
 * allowed (it may synchronise the device). It computes exactly what
 * usp_attn_bwd computes, with the same arguments minus the workspace, and
 * takes its scratch from one fixed 64 MiB array in device memory that the
 * library declares at file scope. It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *  - Arguments are checked first, exactly as usp_attn_bwd checks them
 *    (USP_ERR_INVALID_ARG, USP_ERR_ALIGNMENT, ... before anything else).
 *  - Limit: a problem whose backward scratch (usp_attn_bwd_workspace_size,
 *    B = 1 for packed batches, for the kernels the call would use) exceeds
 *    64 MiB is rejected with USP_ERR_WORKSPACE before anything is launched
 *    (usp_last_error_detail() says why).
 *  - Set-up: the first call on each device (and the first after the
 *    device's context has been reset) looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it. That
 *    lookup is also when the 64 MiB are taken from the device: the array
 *    belongs to a module the CUDA runtime loads on first use (its default,
 *    lazy module loading), and it stays reserved until the process exits.
 *    So make one call on each device before handing the rest of its memory
 *    to a pool and before any stream capture; a call with S = 0 and
 *    otherwise valid sizes (the tensor pointers may then be NULL) does only
 *    this set-up and launches nothing.
 *  - Every call shares the one array, which keeps the last call's contents;
 *    what must start at zero is cleared on the device at the start of each
 *    call. Calls that overlap on the GPU (e.g. on two streams) race on the
 *    array and give wrong results; serialise them.
 * Errors: as usp_attn_bwd, plus USP_ERR_WORKSPACE for the size limit.
 */
usp_status_t usp_attn_bwd_noalloc(const void *q, const void *k, const void *v,
                                  const void *out, const float *lse,
                                  const void *dout, void *dq, void *dk,
                                  void *dv, int B, int S, int Hq, int Hkv,
                                  int D, float softmax_scale, int causal,
                                  int window, int sink_tokens,
                                  const int32_t *cu_seqlens, int cp_size,
                                  int ulysses_degree, usp_layout_t layout,
                                  usp_dtype_t dtype, unsigned flags,
                                  usp_stream_t stream);

/*
 * usp_merge_partials - merge n attention partials with the log-sum-exp rule.
 *
 * "Tree Attention" (Long Context Attention notes): because logsumexp and max
 * are associative, partials over disjoint key sets can be reduced in any
 * order, e.g. a tree. For two partials
 *   L = max + log(exp(L_a - max) + exp(L_b - max)),
 *   O = exp(L_a - L) O_a + exp(L_b - L) O_b;
 * a partial with L = -inf is the identity (its O is ignored).
 *
 * o_parts   [n, rows, D] fp32, lse_parts [n, rows] fp32 (partial i at i*rows)
 * n >= 1 (tree_order: n <= 64), rows >= 0, D in {64, 128}
 * tree_order 0: ((p0 + p1) + p2) + ...   (ring order)
 *            1: pairwise levels (p0+p1), (p2+p3), ...; an odd last partial
 *               moves up a level unchanged.
 * o_out [rows, D] written in out_dtype; lse_out [rows] fp32 written.
 * Errors: USP_ERR_INVALID_ARG, USP_ERR_ALIGNMENT, USP_ERR_CUDA.
 */
usp_status_t usp_merge_partials(const float *o_parts, const float *lse_parts,
                                int n, int64_t rows, int D, int tree_order,
                                void *o_out, usp_dtype_t out_dtype,
                                float *lse_out, usp_stream_t stream);

/*
 * usp_attn_fwd_qkvpacked / usp_attn_bwd_qkvpacked - the same calls on one
 * packed tensor.
 *
 * The YunChang README's LongContextAttentionQKVPacked ("2. Usage"; its
 * benchmark conclusions find the packed form faster) takes q, k and v as one
 * tensor. qkv [B, S, 3, H, D] (rank-major order, as usp_permute(EXTRACT)
 * gives when called with 3*H heads), Hq = Hkv = H: q is qkv[:, :, 0], k
 * qkv[:, :, 1], v qkv[:, :, 2]. Nothing is unpacked: the kernels read the
 * three parts in place with a token stride of 3*H*D elements (and the
 * Ulysses exchange reads them from the packed tensor directly). The
 * backward writes dq, dk, dv into dqkv [B, S, 3, H, D] the same way.
 * out, lse, dout and every other argument, requirement, the workspace (size
 * it with usp_attn_{fwd,bwd}_workspace_size(B, S, H, H, D, ...)) and the
 * errors are those of usp_attn_fwd / usp_attn_bwd.
 */
usp_status_t usp_attn_fwd_qkvpacked(const void *qkv, void *out, float *lse,
                                    int B, int S, int H, int D,
                                    float softmax_scale, int causal, int window,
                                    int sink_tokens, const int32_t *cu_seqlens,
                                    int cp_size, int ulysses_degree,
                                    usp_layout_t layout, usp_dtype_t dtype,
                                    unsigned flags, void *workspace,
                                    size_t workspace_bytes, usp_stream_t stream);

usp_status_t usp_attn_bwd_qkvpacked(const void *qkv, const void *out,
                                    const float *lse, const void *dout,
                                    void *dqkv, int B, int S, int H, int D,
                                    float softmax_scale, int causal, int window,
                                    int sink_tokens, const int32_t *cu_seqlens,
                                    int cp_size, int ulysses_degree,
                                    usp_layout_t layout, usp_dtype_t dtype,
                                    unsigned flags, void *workspace,
                                    size_t workspace_bytes, usp_stream_t stream);

/*
 * usp_attn_fwd_fp8 - usp_attn_fwd on 8-bit float (E4M3) q, k, v.
 *
 * The USP README ("3. Test") runs a forward-only fp8 attention backend
 * under the same sequence-parallel wrappers; the pages give no arithmetic
 * for it. This call computes the attention of usp_attn_fwd (same masks,
 * GQA, varlen, ring schedule, layouts and Ulysses exchange) of the real
 * values e4m3(code) * descale, with one descale per tensor:
 *   s_ij = softmax_scale * <q_i, k_j>   (real values),
 *   O_i = sum_j exp(s_ij - LSE_i) v_j,  LSE_i = log sum_j exp(s_ij).
 * Both products run on the tensor cores on the codes (fp32 accumulation);
 * the probabilities are rounded to E4M3 (as codes of 16 p) for the P V
 * product, which the result's tolerance has to cover; LSE is taken from the
 * unrounded fp32 probabilities.
 *
 * q [B,S,Hq,128], k, v [B,S,Hkv,128]: E4M3 codes (OCP 8-bit float, E4M3:
 *      bias 7, largest finite 448, 0x7F / 0xFF NaN), rank-major as in
 *      usp_attn_fwd (packed [T,H,128] with cu_seqlens), 16-byte aligned.
 * q_descale, k_descale, v_descale  finite, > 0 (else USP_ERR_INVALID_ARG).
 * out  [B,S,Hq,128] bf16, written.  lse  as in usp_attn_fwd.
 * Other arguments as in usp_attn_fwd (dtype is implied; flags: none
 *      apply, USP_FLAG_NATURAL_ORDER gives USP_ERR_UNSUPPORTED).
 * workspace  at least usp_attn_fwd_fp8_workspace_size(...) bytes, 16-byte
 *      aligned, never NULL for S > 0 (it holds V transposed to
 *      [B][Hkv][128][S]); contents on entry irrelevant.
 * Errors: as usp_attn_fwd; USP_ERR_UNSUPPORTED for a head dim other than
 *      128 or a shard / zigzag chunk that is not a multiple of 128 tokens.
 */
usp_status_t usp_attn_fwd_fp8(const void *q, const void *k, const void *v,
                              float q_descale, float k_descale, float v_descale,
                              void *out, float *lse, int B, int S, int Hq, int Hkv,
                              int D, float softmax_scale, int causal, int window,
                              int sink_tokens, const int32_t *cu_seqlens,
                              int cp_size, int ulysses_degree, usp_layout_t layout,
                              unsigned flags, void *workspace, size_t workspace_bytes,
                              usp_stream_t stream);

/* Bytes of scratch usp_attn_fwd_fp8 needs (B: the tensors' batch rows, 1
 * for packed sequences); 0 for invalid sizes. */
size_t usp_attn_fwd_fp8_workspace_size(int B, int S, int Hq, int Hkv, int D,
                                       int cp_size, int ulysses_degree);

/*
 * usp_quantize_e4m3 - out[i] = E4M3 code of x[i] * inv_scale.
 *
 * x  n bf16 values (device, 16-byte aligned); out  n codes (device,
 * 16-byte aligned). The product is taken in fp32 (rounded to nearest) and
 * rounded to the nearest code, ties to the even code; finite values beyond
 * 448 saturate to +-448, NaN stays NaN. The matching descale for
 * usp_attn_fwd_fp8 is 1 / inv_scale. Errors: USP_ERR_INVALID_ARG (n < 0,
 * NULL pointers with n > 0, inv_scale not finite), USP_ERR_ALIGNMENT,
 * USP_ERR_CUDA.
 */
usp_status_t usp_quantize_e4m3(const void *x, void *out, int64_t n, float inv_scale,
                               usp_stream_t stream);

/*
 * usp_attn_decode - one decoding step against a KV cache sharded over a ring.
 *
 * "Long Context Attention" notes, "Ring Attention": flash decoding is ring
 * attention at inference time; "Tree Attention": the partials that the
 * devices compute for a decoding step are combined by a tree reduction
 * (logsumexp is associative). The newest Tq tokens of every sequence attend
 * to all S cached keys; token t sits at position S - Tq + t, and with causal
 * it sees keys j <= S - Tq + t (else all S).
 *
 * q    [B, Tq, Hq, D] bf16;  k, v [B, S, Hkv, D] bf16, the cache in rank-major
 *      contiguous order (rank r's shard is keys [r S/cp, (r+1) S/cp)).
 * out  [B, Tq, Hq, D] bf16;  lse [B, Tq, Hq] fp32 (natural log of the scaled
 *      scores' sum).
 * Every shard is cut into splits_per_shard equal pieces; each piece's partial
 * (O, LSE) is computed separately (fp32, in the workspace) and the
 * cp_size * splits_per_shard partials are merged in key order, pairwise
 * levels (tree_order = 1: a shard's pieces first, then the shards) or left to
 * right (0), as usp_merge_partials does.
 * Requirements: Hq % Hkv == 0, (Hq / Hkv) * Tq <= 16, D in {64, 128},
 * S % (cp_size * splits_per_shard) == 0 and each piece a multiple of 64 keys,
 * Tq <= S, tree_order: cp_size * splits_per_shard <= 64; 16-byte aligned
 * pointers; dtype USP_BF16 (USP_FP32 gives USP_ERR_UNSUPPORTED).
 * workspace: at least usp_attn_decode_workspace_size(...) bytes, 256-byte
 * aligned; its contents on entry are irrelevant.
 * Asynchronous on `stream`. Errors: USP_ERR_INVALID_ARG, USP_ERR_UNSUPPORTED,
 * USP_ERR_ALIGNMENT, USP_ERR_WORKSPACE, USP_ERR_CUDA.
 */
usp_status_t usp_attn_decode(const void *q, const void *k, const void *v,
                             void *out, float *lse, int B, int Tq, int S,
                             int Hq, int Hkv, int D, float softmax_scale,
                             int causal, int cp_size, int splits_per_shard,
                             int tree_order, usp_dtype_t dtype, void *workspace,
                             size_t workspace_bytes, usp_stream_t stream);

size_t usp_attn_decode_workspace_size(int B, int Tq, int S, int Hq, int Hkv,
                                      int D, int cp_size, int splits_per_shard);

/*
 * usp_permute - sequence layouts and the Ulysses all-to-all, bit-exact.
 *
 * EXTRACT / RESTORE (the YunChang README's EXTRACT_FUNC_DICT /
 * zigzag_extract_local reorder, "2. Usage"; stripe and zigzag as in the
 * conventions above):
 *   src/dst [B, S, H, D] (packed: B = 1 and S = T; pass cu_seqlens = NULL,
 *   the layout applies to the packed sequence as a whole).
 *   EXTRACT: dst[b][p] = src[b][pos(p)], RESTORE: dst[b][pos(p)] = src[b][p].
 * ULYSSES_SEQ2HEAD (DeepSpeed-Ulysses exchange inside USP; the degree cannot
 *   exceed the head count, YunChang README): rank w = rho*ud + u sends the
 *   head slice u' of its sequence shard to rank (rho, u'), which stacks the
 *   slices it receives along the sequence in u order. Emulated layout:
 *     src [B, S, H, D] rank-major -> dst [ud, B, S, H/ud, D] with
 *     dst[u][b][p][h][d] = src[b][p][u*H/ud + h][d].
 * ULYSSES_HEAD2SEQ is its inverse (dst [B,S,H,D], src [ud,B,S,H/ud,D]).
 * elem_bytes 1 (E4M3 codes), 2 or 4. H*D*elem_bytes (Ulysses: H/ud*D*elem_bytes) must be a
 * multiple of 16. S divisible as for usp_attn_fwd. src and dst must not
 * overlap. Errors: USP_ERR_INVALID_ARG, USP_ERR_ALIGNMENT, USP_ERR_CUDA.
 */
usp_status_t usp_permute(const void *src, void *dst, usp_permute_kind_t kind,
                         usp_layout_t layout, int B, int S, int H, int D,
                         int cp_size, int ulysses_degree, int elem_bytes,
                         usp_stream_t stream);

/*
 * Kernel timer, for benchmarks and profiling (no counterpart on the pages).
 * While enabled, every kernel this library launches is bracketed by a pair
 * of CUDA events recorded on the launch stream. usp_profile_read() waits
 * for the recorded events, writes one entry per kernel name (launch count
 * and summed device milliseconds) into `stats` (at most max_stats entries),
 * clears the records and returns the number of entries written (negative
 * on a CUDA error). Not thread-safe: enable it only in single-threaded
 * measurement code. The events are created by the CUDA runtime; no device
 * memory is allocated.
 */
typedef struct {
  char name[48];
  uint64_t launches;
  double total_ms;
} usp_kernel_stat_t;

usp_status_t usp_profile_enable(int on);
int usp_profile_read(usp_kernel_stat_t *stats, int max_stats);

/* Waits for the device, then reports (and clears) what the kernels flagged
 * since the last call: USP_ERR_TIMEOUT if a tensor-core kernel gave up on a
 * pipeline wait (each wait is bounded; a kernel that gives up skips its
 * remaining work, frees its tensor memory and exits, leaving its outputs
 * unspecified), USP_ERR_CUDA if the device reports an error or a kernel
 * found its launch environment unusable (a shared-memory window without the
 * 1024-byte alignment its swizzled tiles need; it then did nothing), else
 * USP_OK.
 * Synchronises the whole device: a diagnostics call, not for hot loops. */
usp_status_t usp_device_status(void);

/*
 * usp_selftest_wait_timeout - exercise the failure path of usp_device_status.
 *
 * A diagnostics call with no counterpart on the pages. It launches one small
 * kernel whose pipeline wait (the same bounded mbarrier wait the attention
 * kernels use) waits on a phase that nothing ever completes. After limit_us
 * microseconds (1 .. 1000000) the wait gives up, records USP_ERR_TIMEOUT in
 * a device status word and the kernel exits normally: the next
 * usp_device_status() then returns USP_ERR_TIMEOUT (and clears it), and the
 * device stays usable. Nothing faults or traps. Asynchronous on `stream`.
 * Errors: USP_ERR_INVALID_ARG (limit out of range), USP_ERR_CUDA.
 */
usp_status_t usp_selftest_wait_timeout(unsigned limit_us, usp_stream_t stream);

/* Which CUDA call failed, and why, for the last USP_ERR_CUDA returned on the
 * calling thread, or why an argument was refused where a call's description
 * says so (thread-local storage, never NULL; empty if none). */
const char *usp_last_error_detail(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char *usp_status_string(usp_status_t status);

/* Number of kernel launches this library has enqueued in the calling
 * process so far (host-side counter; for launch accounting). */
uint64_t usp_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* USP_H_ */
