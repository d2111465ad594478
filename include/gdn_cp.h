/*
 * gdn_cp.h -- C ABI of the context-parallel Gated DeltaNet forward for one
 * NVIDIA GB300 (sm_103a).
 *
 * What it computes (sources are two public web pages):
 *   [FLA-CP] flash-linear-attention, fla/ops/cp/context.py: get_cp_cu_seqlens
 *            and build_cp_context (the per-shard cu_seqlens plan).
 *   [HP-CP]  hyper-parallel, linear_attention_context_parallel.py: the causal
 *            conv1d + SiLU with the previous shard's halo
 *            (_causal_conv1d_with_cp_halo), the chunked gated delta rule in
 *            WY/UT form (_prepare_gdn_chunks_for_summary,
 *            _run_prepared_gdn_chunks), the shard state summary
 *            (_compute_gdn_state_summary_from_prepared) and its prefix merge
 *            (_merge_gdn_prefix_state_summaries_torch).
 *
 * The gated delta rule, per sequence and value head, with S a [dk, dv] fp32
 * state:   S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *          o_t = S_t^T (scale q_t)
 * A long sequence may be cut into P contiguous "virtual shards" of one
 * device's memory; each shard's state map S_out = M S_in + N is combined by
 * a prefix scan so that the sharded result equals the unsharded one.
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" must be CUDA device (or managed) memory; the
 *     caller allocates and owns every buffer.  Except for the workspaces of
 *     gdn_shard_fwd (required) and gdn_chunk_fwd (optional), no entry point
 *     needs scratch memory, and none allocates.
 *   - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL
 *     = the legacy default stream).  No entry point synchronises the host.
 *   - Tokens are packed, batch 1: a token-major [T, ...] layout with
 *     sequence boundaries in cu_seqlens (int32, device, [num_seqs + 1],
 *     cu_seqlens[0] = 0, non-decreasing, cu_seqlens[num_seqs] = T).
 *     Empty sequences are allowed.
 *   - Head layout: Hk query/key heads, Hv value heads, Hv % Hk == 0; value
 *     head h reads query/key head h / (Hv / Hk) (repeat_interleave on the
 *     head dimension, [HP-CP] the P2P wrapper's forward).
 *   - Supported: dk, dv in {32, 64, 128}; conv kernel size 1..4; chunk 64.
 *   - dtype GDN_BF16: q/k/v/x/beta/o/conv weights in bf16, arithmetic and
 *     the state in fp32.  GDN_F32: everything fp32.  g is always fp32.
 *   - Errors detectable on the host return a non-OK status before anything
 *     is enqueued; gdn_last_error() then describes the first failing check.
 *     Errors that depend on device data (a malformed cu_seqlens) are written
 *     to a device status word (see gdn_cp_plan) and never trap.
 */
#ifndef GDN_CP_H
#define GDN_CP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,       /* null pointer, negative size, misaligned buffer */
    GDN_ERR_UNSUPPORTED_SHAPE = 2, /* dk/dv/conv_k/channels outside the supported set */
    GDN_ERR_DTYPE = 3,             /* unknown gdn_dtype */
    GDN_ERR_NOT_DIVISIBLE = 4,     /* T % n_shards != 0 ([HP-CP] _slice_local_cp) */
    GDN_ERR_SHARD_TOO_SHORT = 5,   /* T / n_shards < conv_k - 1 ([HP-CP] conv halo check) */
    GDN_ERR_BAD_CU_SEQLENS = 6,    /* device status only: cu_seqlens malformed */
    GDN_ERR_TIMEOUT = 7,           /* device status only: a bounded wait expired */
    GDN_ERR_CUDA = 8,              /* a CUDA launch failed; see gdn_last_error() */
    GDN_ERR_WORKSPACE = 9          /* workspace missing or smaller than required */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* flags for gdn_chunk_fwd / gdn_chunk_summary / gdn_shard_fwd */
enum {
    /* replace q and k by x * rsqrt(sum(x^2) + 1e-6) per head before use
       ([HP-CP] _l2norm_torch, use_qk_l2norm_in_kernel) */
    GDN_QK_L2NORM = 1u
};

/* Human-readable name of a status code (static string). */
const char *gdn_status_string(gdn_status s);

/* Thread-local description of the last non-OK status returned on this
   thread ("" if none). */
const char *gdn_last_error(void);

/* Number of bounded device-side waits (on the tensor core) that expired on
   the current device since load or the last reset; such a wait makes its
   kernel stop early and leave its outputs incomplete.  Synchronises the
   device (a copy from device memory).  reset != 0 zeroes the counter. */
gdn_status gdn_device_timeouts(int32_t *count, int reset);

/* Testing hook (no counterpart on the source pages): settings of the
   split-item hand-over of the tensor-core chunk kernel, used by the launches
   that follow on any thread.  wait_ns bounds the wait of a second half for
   its first half's final state (default 1e9 ns); publish == 0 makes first
   halves skip publishing it, so that every second half's wait expires:
   the kernel then stops early, counts a timeout (gdn_device_timeouts) and
   writes GDN_ERR_TIMEOUT to the launch's status word (the plan's word for
   gdn_shard_fwd, word 2 of the gdn_chunk_fwd workspace).  Restore with
   gdn_debug_set_handover(1000000000, 1).  Not for production use. */
gdn_status gdn_debug_set_handover(int64_t wait_ns, int publish);

/* Testing hook (no counterpart on the source pages): enable = 0 turns off the
   splitting of work-queue items into two parts handed over through a final
   state (single-segment launches: long items in halves; shard passes: short
   tail parts), so that a test can compare split and unsplit runs, which give
   bit-identical results.  enable = 1 (the default) restores it.  Applies to
   launches made after the call from any thread.  Not for production use. */
gdn_status gdn_debug_set_split(int32_t enable);

/* Profiling hook (no counterpart on the source pages): while n > 0, every
   gdn_shard_fwd call on this host thread records events[i] (cudaEvent_t
   handles, created by the caller) on its stream: [0] at entry, [1] after the
   plan and the conv, [2] after chunk pass 1, [3] after the merge, [4] after
   pass 2, [5] at exit (as far as n reaches).  n = 0 turns it off. */
gdn_status gdn_debug_set_phase_events(void *const *events, int32_t n);

/* ------------------------------------------------------------------------
 * Shard plan  ([FLA-CP] get_cp_cu_seqlens, steps 1-5)
 *
 * For each shard r < n_shards (part = T / n_shards, rs = r * part,
 * re = rs + part, cu = cu_seqlens):
 *   s = #{i : cu[i+1] <= rs}            start_seq_idx (searchsorted right)
 *   e = #{i < num_seqs : cu[i] < re}    end_seq_idx   (searchsorted left)
 *   local_cu = dedupe(clamp(cu[s..e], rs, re) - rs)   (unique_consecutive)
 *   pre_num_conv_tokens = max(0, rs - cu[s])
 *   pre_num_ranks  = r - cu[s] / part;        is_first_rank = (pre == 0)
 *   post_num_ranks = (cu[e] - 1) / part - r;  is_last_rank  = (post == 0)
 *
 * `plan` is a device int32 buffer of gdn_cp_plan_words(num_seqs, n_shards)
 * words, laid out as:
 *   plan[0]                                  status word (0 = OK, else a
 *                                            gdn_status: BAD_CU_SEQLENS when
 *                                            cu[0] != 0, cu decreases, or
 *                                            cu[num_seqs] % n_shards != 0)
 *   plan[GDN_PLAN_REC(r) + GDN_PLAN_*]       the fields below for shard r
 *   plan[GDN_PLAN_CU(num_seqs, n_shards, r) + i], 0 <= i <= local_num_seqs
 *                                            local cu_seqlens of shard r
 *   plan[GDN_PLAN_SEQ(num_seqs, n_shards, r) + j], 0 <= j < local_num_seqs
 *                                            global index of the sequence that
 *                                            local segment j belongs to (the one
 *                                            holding the segment's first token;
 *                                            empty sequences, which the dedupe
 *                                            of step 4 removes, own no segment)
 * Needs 1 <= n_shards <= 65536 and num_seqs >= 1.  The whole plan is
 * computed on the device: no device-to-host copy of cu_seqlens.
 * ---------------------------------------------------------------------- */
enum {
    GDN_PLAN_LOCAL_NUM_SEQS = 0,
    GDN_PLAN_START_SEQ_IDX = 1,
    GDN_PLAN_END_SEQ_IDX = 2,
    GDN_PLAN_PRE_NUM_RANKS = 3,
    GDN_PLAN_POST_NUM_RANKS = 4,
    GDN_PLAN_IS_FIRST_RANK = 5,
    GDN_PLAN_IS_LAST_RANK = 6,
    GDN_PLAN_PRE_NUM_CONV_TOKENS = 7,
    GDN_PLAN_SEG_OFFSET = 8, /* sum of local_num_seqs over shards < r */
    GDN_PLAN_NFIELDS = 9
};
#define GDN_PLAN_REC(r) (1 + (int64_t)(r) * GDN_PLAN_NFIELDS)
#define GDN_PLAN_CU(num_seqs, n_shards, r) \
    (1 + (int64_t)(n_shards) * GDN_PLAN_NFIELDS + (int64_t)(r) * ((num_seqs) + 1))
#define GDN_PLAN_SEQ(num_seqs, n_shards, r) \
    (GDN_PLAN_CU(num_seqs, n_shards, n_shards) + (int64_t)(r) * ((num_seqs) + 1))

int64_t gdn_cp_plan_words(int32_t num_seqs, int32_t n_shards);

gdn_status gdn_cp_plan(const int32_t *cu_seqlens, int32_t num_seqs, int32_t n_shards,
                       int32_t *plan, void *stream);

/* ------------------------------------------------------------------------
 * Causal depthwise conv1d + SiLU with a halo
 * ([HP-CP] _causal_conv1d_with_cp_halo; zero history before each sequence
 * start, as the varlen plan's pre_num_conv_tokens implies)
 *
 *   y[t, c] = silu(bias[c] + sum_{j < conv_k} w[c, j] * x'[t - conv_k + 1 + j, c])
 *
 * x' is x within the token's own sequence and 0 before its start, except
 * that the FIRST sequence continues from `halo`: halo is [conv_k - 1,
 * channels] (row stride `channels`), its last row being the token just
 * before x[0]; only its last `halo_len` rows are history (0 <= halo_len <=
 * conv_k - 1; halo may be NULL when halo_len == 0).
 *   x     device [T, channels] dtype, row stride ldx (elements)
 *   w     device [channels, conv_k] dtype;  bias device [channels] or NULL
 *   y     device [T, channels] dtype, row stride ldy; must not overlap x
 * Needs channels % 8 == 0, ldx and ldy multiples of 8, and 16-byte aligned
 * x, y and halo.  Accumulates in fp32; bf16 output rounds to nearest even
 * (its SiLU uses a hardware tanh, error about 5e-4, below bf16 rounding;
 * fp32 output uses a / (1 + e^-a)).
 * ---------------------------------------------------------------------- */
gdn_status gdn_conv_silu(const void *x, int64_t ldx, gdn_dtype dtype, int32_t T,
                         int32_t channels, const void *w, const void *bias, int32_t conv_k,
                         const int32_t *cu_seqlens, int32_t num_seqs, const void *halo,
                         int32_t halo_len, void *y, int64_t ldy, void *stream);

/* ------------------------------------------------------------------------
 * Chunked (C = 64) gated delta rule forward, WY/UT form
 * ([HP-CP] _prepare_gdn_chunks_for_summary + _run_prepared_gdn_chunks)
 *
 *   q, k  device [T, Hk, dk] dtype at q + t*ldq + h*dk + i (same for k)
 *   v     device [T, Hv, dv] dtype at v + t*ldv + h*dv + j
 *   g     device [T, Hv] fp32 log-gates (per-token decay exp(g))
 *   beta  device [T, Hv] dtype
 *   h0    device [num_seqs, Hv, dk, dv] fp32 initial states, or NULL (= 0)
 *   o     device [T, Hv, dv] dtype (dense)
 *   h_final device [num_seqs, Hv, dk, dv] fp32 state after each sequence's
 *         last token (h0 or 0 for an empty sequence), or NULL
 *   scale multiplies q (1/sqrt(dk) in the pages)
 *   workspace, workspace_bytes  optional device scratch of at least
 *         gdn_chunk_fwd_workspace_size(...) bytes, 16-byte aligned (the work
 *         queue described there), or NULL, 0
 * Chunks restart at every sequence start; a sequence's last chunk is padded
 * with beta = 0, g = 0 rows that are never stored.  Row strides must be
 * multiples of 8 elements and q/k/v 16-byte aligned.  o may not alias the
 * inputs.
 * ---------------------------------------------------------------------- */
gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v, int64_t ldq,
                         int64_t ldk, int64_t ldv, gdn_dtype dtype, const float *g,
                         const void *beta, const float *h0, const int32_t *cu_seqlens,
                         int32_t num_seqs, int32_t T, int32_t Hk, int32_t Hv, int32_t dk,
                         int32_t dv, float scale, uint32_t flags, void *o, float *h_final,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of the optional gdn_chunk_fwd workspace (device, 16-byte aligned,
 * contents on entry irrelevant; the call rewrites it on its stream).  With a
 * workspace, the bf16 d=128 kernel takes its (sequence, head) jobs from a
 * work queue sorted longest-first, one persistent block per SM; with h_final
 * as well it may split a long sequence's token range into two halves run one
 * after the other (the second starts from the first's final state, handed
 * over through h_final), so that the work packs more evenly onto the SMs.
 * Results are bit-identical with and without a workspace.  Without one every
 * block runs one job, longest first.  A workspace smaller than this size is
 * an error (GDN_ERR_WORKSPACE). */
size_t gdn_chunk_fwd_workspace_size(int32_t num_seqs, int32_t Hv, int32_t dk, int32_t dv,
                                    gdn_dtype dtype);

/* ------------------------------------------------------------------------
 * Head-major layout ([HP-CP] LinearAttentionUlyssesCPWrapper: after its
 * seq-to-heads all-to-all every rank holds whole sequences of a subset of the
 * heads; on one device that exchange is a re-layout of whole d-element rows)
 *   gdn_to_head_major   x device [T, H, d] dtype with token stride ldx
 *                       (elements, ldx >= H*d, 16-byte rows) -> y device
 *                       [H, T, d] dense
 *   gdn_to_token_major  the inverse: y [H, T, d] -> x [T, H, d] (stride ldx)
 *   gdn_chunk_fwd_heads gdn_chunk_fwd on dense head-major q, k [Hk, T, dk],
 *                       v [Hv, T, dv] -> o [Hv, T, dv]; g, beta [T, Hv], h0,
 *                       h_final, cu_seqlens, scale, flags and the optional
 *                       workspace as in gdn_chunk_fwd (same size); q, k, v, o
 *                       16-byte aligned.  Same arithmetic as the token-major
 *                       call, so the results are bit-identical.
 * ---------------------------------------------------------------------- */
gdn_status gdn_to_head_major(const void *x, int64_t ldx, gdn_dtype dtype, int32_t T, int32_t H,
                             int32_t d, void *y, void *stream);
gdn_status gdn_to_token_major(const void *y, gdn_dtype dtype, int32_t T, int32_t H, int32_t d,
                              void *x, int64_t ldx, void *stream);
gdn_status gdn_chunk_fwd_heads(const void *q, const void *k, const void *v, gdn_dtype dtype,
                               const float *g, const void *beta, const float *h0,
                               const int32_t *cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                               int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                               void *o, float *h_final, void *workspace, size_t workspace_bytes,
                               void *stream);

/* ------------------------------------------------------------------------
 * State summary of each sequence ([HP-CP]
 * _compute_gdn_state_summary_from_prepared): the affine map of the state
 * across the sequence,  S_end = M S_start + N, with
 *   M = prod_t exp(g_t) (I - beta_t k_t k_t^T)   device [num_seqs, Hv, dk, dk] fp32
 *   N = the state reached from S_start = 0       device [num_seqs, Hv, dk, dv] fp32
 * computed chunk by chunk on the augmented state [N | M] from [0 | I].
 * Inputs as in gdn_chunk_fwd (q is not needed).
 * ---------------------------------------------------------------------- */
gdn_status gdn_chunk_summary(const void *k, const void *v, int64_t ldk, int64_t ldv,
                             gdn_dtype dtype, const float *g, const void *beta,
                             const int32_t *cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                             int32_t Hv, int32_t dk, int32_t dv, uint32_t flags, float *M,
                             float *N, void *stream);

/* ------------------------------------------------------------------------
 * Prefix merge of shard summaries ([HP-CP]
 * _merge_gdn_prefix_state_summaries_torch), for every value head h:
 *   S_in[0] = S0 (or 0);   S_in[r] = M[r-1] S_in[r-1] + N[r-1],  r = 1..P-1
 *   M device [P, Hv, dk, dk] (16-byte aligned), N device [P, Hv, dk, dv],
 *   S0 device [Hv, dk, dv] or NULL, S_in device [P, Hv, dk, dv]; all fp32.
 *   M[P-1], N[P-1] unused.
 * Sequential over r in fp32, parallel over heads and 32-column tiles of the
 * state; each M is staged in shared memory while the previous one is applied.
 * ---------------------------------------------------------------------- */
gdn_status gdn_state_combine(const float *M, const float *N, const float *S0, int32_t P,
                             int32_t Hv, int32_t dk, int32_t dv, float *S_in, void *stream);

/* ------------------------------------------------------------------------
 * The whole path on P virtual shards of one device:
 *   plan -> conv + SiLU (halo = previous shard's rows) -> q/k/v views of the
 *   conv output -> chunked gated delta rule per shard (pass 1; shards that
 *   continue a sequence from an earlier shard run the [N | M] summary) ->
 *   prefix merge -> pass 2 for the continuing shards.
 *   x       device [T, Cch] dtype, Cch = 2*Hk*dk + Hv*dv, fused channel order
 *           [Q (Hk*dk) | K (Hk*dk) | V (Hv*dv)] ([HP-CP] torch.split of
 *           mixed_qkv); row stride Cch
 *   conv_w  device [Cch, conv_k] dtype; conv_b device [Cch] dtype or NULL
 *   g, beta, h0, o, h_final as in gdn_chunk_fwd
 *   plan_out  device int32 [gdn_cp_plan_words(num_seqs, n_shards)] or NULL:
 *           receives a copy of the plan (incl. its status word)
 *   workspace device, >= gdn_shard_fwd_workspace_size(...) bytes, 256-byte
 *           aligned; its contents on entry do not matter.  For bf16 with
 *           dk = dv = 128 and n_shards > 1 that size includes room in which
 *           the summaries' N halves store their chunks' W rows, K~ tiles and
 *           e^{G_last} (about T * Hv * 512 bytes), so that the M halves run apart on
 *           the tensor cores (with few long shards each M chain is cut into
 *           up to 8 segments, whose fp32 products take n_shards * Hv * 64 KiB
 *           per segment more); a workspace down to
 *           gdn_shard_fwd_workspace_min_size(...) bytes is accepted as well,
 *           with the M halves run in the chunk kernel (the same results up to
 *           rounding; bit for bit where the chains are not cut; slower).  The
 *           size depends on the current device's SM count.
 * With n_shards == 1 this is the ordinary (unsharded) forward.  Checks on
 * the host: T % n_shards == 0 and T / n_shards >= conv_k - 1.  A malformed
 * cu_seqlens sets the plan status word and every later kernel returns
 * without touching o / h_final.
 * ---------------------------------------------------------------------- */
size_t gdn_shard_fwd_workspace_size(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk,
                                    int32_t Hv, int32_t dk, int32_t dv, gdn_dtype dtype);
/* the smallest workspace gdn_shard_fwd accepts (see its workspace argument);
 * 0 for invalid arguments */
size_t gdn_shard_fwd_workspace_min_size(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk,
                                        int32_t Hv, int32_t dk, int32_t dv, gdn_dtype dtype);

gdn_status gdn_shard_fwd(const void *x, const void *conv_w, const void *conv_b, int32_t conv_k,
                         const float *g, const void *beta, const float *h0,
                         const int32_t *cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                         int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                         int32_t n_shards, gdn_dtype dtype, void *workspace,
                         size_t workspace_bytes, void *o, float *h_final, int32_t *plan_out,
                         void *stream);

/* ------------------------------------------------------------------------
 * The layer between its projections ([HP-CP] LinearAttentionP2PCPWrapper /
 * LinearAttentionAllGatherCPWrapper forward, from the projection outputs to
 * the input of the output projection):
 *   beta = sigmoid(b),  g = -exp(A_log) * softplus(a + dt_bias)   (per v-head)
 *   o    = the path of gdn_shard_fwd on n_shards virtual shards
 *   y    = norm_w * o / sqrt(mean(o^2) + norm_eps) * silu(z)   per (token,
 *          v-head) row of dv values (the wrappers' norm(core_attn_out, z))
 *   x, conv_w, conv_b, h0, cu_seqlens, workspace, h_final, plan_out: as in
 *           gdn_shard_fwd (same workspace size)
 *   a, b    device [T, Hv] dtype (the raw gate projections)
 *   A_log, dt_bias  device [Hv] fp32
 *   z       device [T, Hv, dv] dtype with token row stride ldz (a multiple of
 *           8, >= Hv*dv), 16-byte aligned; or NULL: no norm (y = o)
 *   norm_w  device [dv] dtype, 16-byte aligned (with z)
 *   y       device [T, Hv, dv] dtype
 * The gates are computed where g and beta are read (inside the chunk
 * kernels): g in fp32 (softplus(x) = x for x > 20), beta rounded to dtype.
 * The norm is the tensor-core chunk kernel's output epilogue for bf16 with
 * dk = dv = 128 (on the bf16-rounded o); other shapes run it as one more
 * pass over y.
 * ---------------------------------------------------------------------- */
gdn_status gdn_layer_fwd(const void *x, const void *conv_w, const void *conv_b, int32_t conv_k,
                         const void *a, const void *b, const float *A_log, const float *dt_bias,
                         const void *z, int64_t ldz, const void *norm_w, float norm_eps,
                         const float *h0, const int32_t *cu_seqlens, int32_t num_seqs, int32_t T,
                         int32_t Hk, int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                         int32_t n_shards, gdn_dtype dtype, void *workspace, size_t workspace_bytes,
                         void *y, float *h_final, int32_t *plan_out, void *stream);

/* ------------------------------------------------------------------------
 * Backward of the gated delta rule ([HP-CP] the custom autograd functions
 * _RecvInitialStateP2PFunction / _SendFinalStateP2PFunction, whose backward
 * sends the state gradient the other way; the forward is gdn_chunk_fwd's).
 * Given the loss gradients dout (w.r.t. o) and dh_final (w.r.t. the final
 * states), computes the gradients w.r.t. every input of gdn_chunk_fwd:
 *   per token, with a = e^g, P = a S_prev, u = v - P^T k, S = P + beta k u^T,
 *   o = S^T (scale q), walked backwards with the state gradient dS:
 *     dq = scale S do,  dS += scale q do^T,  dbeta = k . (dS u),
 *     du = beta dS^T k = dv,  dk = beta dS u - P du,  dP = dS - k du^T,
 *     dg = <P, dP>,  dS_prev = a dP;   dh0 = dS before the first token.
 *   q, k, v, ldq, ldk, ldv, dtype, g, beta, h0, cu_seqlens, num_seqs, T, Hk,
 *           Hv, dk, dv, scale, flags: as in gdn_chunk_fwd (the same forward)
 *   dout    device [T, Hv, dv] dtype, dense
 *   dh_final device [num_seqs, Hv, dk, dv] fp32, or NULL (zero)
 *   dq, dk_ device [T, Hk, dk] fp32 (summed over the Hv/Hk value heads that
 *           read the q/k head; gradients of the stored q, k, through the L2
 *           norm when flags has GDN_QK_L2NORM)
 *   dv_     device [T, Hv, dv] fp32;  dg, dbeta device [T, Hv] fp32
 *   dh0     device [num_seqs, Hv, dk, dv] fp32 (also when h0 is NULL)
 *   workspace device, >= gdn_chunk_bwd_workspace_size(...) bytes, 256-byte
 *           aligned, contents on entry irrelevant (8-token block-start states of every
 *           sequence and a per-(sequence, head) replay scratch)
 * dk, dv in {32, 64, 128}.  One block of 512 threads per (sequence, value
 * head); the states before each token are recomputed from block-start
 * checkpoints, so the cost grows with the longest sequence.
 * ---------------------------------------------------------------------- */
size_t gdn_chunk_bwd_workspace_size(int32_t T, int32_t num_seqs, int32_t Hk, int32_t Hv, int32_t dk,
                                    int32_t dv);
gdn_status gdn_chunk_bwd(const void *q, const void *k, const void *v, int64_t ldq, int64_t ldk,
                         int64_t ldv, gdn_dtype dtype, const float *g, const void *beta,
                         const float *h0, const void *dout, const float *dh_final,
                         const int32_t *cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                         int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags, float *dq,
                         float *dk_, float *dv_, float *dg, float *dbeta, float *dh0,
                         void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * gdn_chunk_bwd with every sequence cut into its pieces on n_shards virtual
 * shards ([HP-CP] the backward of _RecvInitialStateP2PFunction /
 * _SendFinalStateP2PFunction: the state gradient travels from a shard to the
 * one before it).  The pieces (the shard plan's local segments) run in
 * parallel: each piece's state map S_end = M S_start + N comes from its
 * summary, the start states from a forward merge over each sequence's pieces,
 * each piece's start-state gradient from its own outputs (b) from a first
 * backward pass, the end-state gradients from the reverse merge
 * dS_end(j - 1) = M_j^T dS_end(j) + b_j (dS_end of a sequence's last piece =
 * dh_final), and the input gradients from a second backward pass.
 * Arguments and results as in gdn_chunk_bwd, plus:
 *   n_shards  1..65536, T % n_shards == 0
 *   workspace device, >= gdn_shard_bwd_workspace_size(...) bytes, 256-byte
 *             aligned, contents on entry irrelevant
 *   plan_out  device int32 [gdn_cp_plan_words(num_seqs, n_shards)] or NULL:
 *             receives the shard plan; its status word is
 *             GDN_ERR_BAD_CU_SEQLENS when cu_seqlens is malformed, in which
 *             case no gradient beyond zeroed dq / dk is written
 * Results equal gdn_chunk_bwd's up to rounding.
 * ---------------------------------------------------------------------- */
size_t gdn_shard_bwd_workspace_size(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk,
                                    int32_t Hv, int32_t dk, int32_t dv);
gdn_status gdn_shard_bwd(const void *q, const void *k, const void *v, int64_t ldq, int64_t ldk,
                         int64_t ldv, gdn_dtype dtype, const float *g, const void *beta,
                         const float *h0, const void *dout, const float *dh_final,
                         const int32_t *cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                         int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                         int32_t n_shards, float *dq, float *dk_, float *dv_, float *dg,
                         float *dbeta, float *dh0, void *workspace, size_t workspace_bytes,
                         int32_t *plan_out, void *stream);

/* ------------------------------------------------------------------------
 * gdn_shard_fwd without a caller workspace.  The source pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- a plugin whose host application owns all device buffers
 * and passes it only inputs and outputs, or a latency-critical loop that may
 * not call cudaMalloc (which can synchronise the device).
 *
 * Same arguments and results as gdn_shard_fwd, minus the workspace.  The
 * scratch is one file-scope device array of GDN_NOALLOC_SCRATCH_BYTES
 * (32 MiB) that every device loading the library holds until the process
 * exits.  A problem whose gdn_shard_fwd_workspace_min_size(...) exceeds it is
 * rejected with GDN_ERR_WORKSPACE before anything is enqueued.  The entry
 * point never calls cudaMalloc/cudaFree or any allocating routine.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it with
 *     the device's current CUDA context; a call under a new context (after
 *     cudaDeviceReset) looks it up again.  Make the first call on a device,
 *     and the first after a reset, before any stream capture.
 *   - All calls share the one array and it keeps the previous call's
 *     contents; nothing in it needs to start at zero.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on it:
 *     serialise them, e.g. on one stream.
 * ---------------------------------------------------------------------- */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)

gdn_status gdn_shard_fwd_noalloc(const void *x, const void *conv_w, const void *conv_b,
                                 int32_t conv_k, const float *g, const void *beta, const float *h0,
                                 const int32_t *cu_seqlens, int32_t num_seqs, int32_t T,
                                 int32_t Hk, int32_t Hv, int32_t dk, int32_t dv, float scale,
                                 uint32_t flags, int32_t n_shards, gdn_dtype dtype, void *o,
                                 float *h_final, int32_t *plan_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_CP_H */
