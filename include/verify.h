/*
 * verify.h -- C ABI of libverify: the weight-streaming verify pass of speculative decoding on one
 * NVIDIA GB300 (sm_103a).
 *
 * One verify pass streams every weight of a 64-layer hybrid target once for M = 8 * lanes rows
 * (per lane: the committed anchor token and 7 draft tokens; 1..4 lanes).  Sources, by page title and
 * section:
 *   [LM-bus]     "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max",
 *                section "What one token costs the bus" (NVFP4 MLP + FP8 E4M3 mixer projections +
 *                NVFP4 head = the bytes read on every pass; tensor-group table).
 *   [LM-formats] same page, section "Formats, and what runs where" (NVFP4 = E2M1 codes, one E4M3
 *                scale per 16 weights, an FP32 tensor scale that MULTIPLIES; scale codes top out at
 *                448; weight-only arithmetic: BF16 activations, FP32 accumulation).
 *   [LM-accept]  same page, section "The megakernel is per layer, not per step" (greedy acceptance:
 *                accept the longest prefix of drafts equal to the target's tokens, commit the
 *                target's token after it; 1..8 tokens per round).
 *   [SP-geom]    "144 tok/s needs 502 GB/s" (Splash), sections "The engine hard-codes the model"
 *                (geometry; nine bytes per sixteen weights) and "The decode step is one command
 *                buffer" (8 verify rows per lane, up to 4 lanes, one submission per step).
 *   [BS-ties]    "Beating Splash on an M5 Max", section "The bugs a second reviewer found" (GPU and
 *                CPU must break argmax ties the same way) and "The kernels were not the gap"
 *                (split-K for narrow projections).
 *   [SP-sample]  "144 tok/s needs 502 GB/s" (Splash), section "Exact, up to top-32" (standard
 *                speculative sampling, accept when u * q < p, else draw from max(p - q, 0); the
 *                target's probabilities are temperature over its first top_k <= 32 entries,
 *                truncated by top_p, renormalised); "lithos-metal ...", section "How DSpark is wired
 *                in" (a greedy drafter is a point mass); "Beating Splash on an M5 Max", section "What
 *                actually moved the needle" (one GPU kernel over the verify logits applies top-k and
 *                top-p, samples and runs the acceptance rule).
 *   [LM-attn]    "lithos-metal ...", section "The megakernel is per layer, not per step" (the full-
 *                attention figure and text: an attention core that reads and appends a BF16 KV cache,
 *                causal softmax of q k^T weighting V, times the sigmoid of the gate; the KV range split
 *                into partitions of up to 1,024 keys whose online-softmax partials are merged).
 *   [BS-gdn]     "Beating Splash on an M5 Max", section "What actually moved the needle" (the GDN step
 *                writes out of place from parity buffer A to B; a partly rejected round re-scans only
 *                the committed rows from the intact A; the state after every possible number of kept
 *                tokens matches a reference scan exactly); "lithos-metal ...", sections "What one
 *                token costs the bus" (fp32 state (v_heads, dk, dv) = 48 x 128 x 128 per layer) and
 *                "The megakernel is per layer, not per step" (the commit re-scan).
 *   [LOOP]       "lithos-metal ...", section "What one token costs the bus" (the embedding is a gather
 *                of the 4-bit table); "Speculative decoding" (mlx-dspark), sections "Lookup (no
 *                drafter)" and "Lookup drafts" (the continuation of an earlier match of the current
 *                text is a free draft); "Beating Splash on an M5 Max", section "The kernels were not
 *                the gap" (host synchronisations per round were the cost).
 *   [WIDE]       "Speculative decoding" (mlx-dspark), section "Lookup drafts": when the current text's
 *                match runs deep, drafts grow (to 32 tokens) and 16-32 rows are verified in one pass;
 *                the acceptance rule is the same longest prefix [LM-accept] over R - 1 drafts.
 *   [SP-q4]      "144 tok/s needs 502 GB/s" (Splash), section "The engine hard-codes the model": the
 *                other engines' affine 4-bit format, per group of 64 inputs 32 bytes of codes plus
 *                a bf16 scale and a bf16 bias (nine bytes per sixteen weights); "Beating Splash on
 *                an M5 Max", section "What actually moved the needle" (the Q4 tiles use per-group
 *                input sums).
 *
 * Conventions for every entry point:
 *   - Device pointers are plain CUDA device addresses owned by the caller; the library never
 *     allocates or frees device memory and never keeps a pointer beyond the call, except a
 *     vp_model, which stores the weight pointers given to vp_model_create (the caller keeps them
 *     alive and unchanged while the model is used).
 *   - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream); no call synchronises the host.  vp_verify_pass issues no host synchronisation and
 *     no allocation, so it can be captured into a CUDA graph.
 *   - Arguments are validated on the host before any launch; an invalid call returns an error and
 *     enqueues nothing.  The library never aborts, throws or prints.
 *   - Workspace: `ws` is caller-owned device memory of at least vp_*_workspace_bytes() bytes,
 *     256-byte aligned, zero-filled once before its first use (vp_workspace_init).  The kernels
 *     leave the counters they use back at zero, so a call that completes normally leaves the
 *     workspace ready for the next call without any per-call reset (each call is a pure sequence
 *     of kernel launches).  The first 4 bytes hold a sticky device status word: 0, or
 *     VP_ERR_TIMEOUT once a bounded device-side wait gave up (then re-initialise the workspace).
 *     Read it after the stream has synchronised (vp_read_status).  Calls that share a workspace
 *     must be ordered on one stream.
 *   - Inputs are read-only; outputs are fully overwritten.
 */
#ifndef VERIFY_H_
#define VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VP_OK = 0,
  VP_ERR_INVALID_ARG = 1, /* null pointer, negative size, unknown enum */
  VP_ERR_SHAPE = 2,       /* unsupported M, N or K (see each call) */
  VP_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned (workspace: 256-byte) */
  VP_ERR_WORKSPACE = 4,   /* ws_bytes smaller than the matching vp_*_workspace_bytes() */
  VP_ERR_CUDA = 5,        /* a CUDA runtime call failed; vp_get_last_cuda_error() has the code */
  VP_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up (reported in the status word) */
  VP_ERR_UNSUPPORTED = 7  /* no sm_103a device, or an unsupported configuration */
} vp_status;

/* Human-readable name of a status code (static string). */
const char* vp_status_string(int status);

/* The CUDA error code of the most recent VP_ERR_CUDA on the calling thread (0 if none). */
int vp_get_last_cuda_error(void);

/* Zero-fills ws_bytes of the workspace on `stream` (required once before first use, and after
 * an error). */
vp_status vp_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Copies the device status word at the start of `ws` to *status (synchronous: it waits for
 * `stream`).  Returns VP_OK or VP_ERR_CUDA. */
vp_status vp_read_status(const void* ws, int* status, void* stream);

/* ------------------------------------------------------------------ packed weight layouts
 *
 * Canonical (logical) layouts, row-major [N][K] as in nn.Linear:
 *   NVFP4: codes [N][K/2] bytes, element 2j of a row is the LOW nibble of byte j; each nibble is an
 *          E2M1 code (bit 3 sign, bits 2..1 exponent, bit 0 mantissa); scales [N][K/16] E4M3 (FN)
 *          bytes, scale[n][k/16] applies to weights k..k+15 of row n.  [LM-formats]
 *   FP8:   [N][K] E4M3 (FN) bytes, one fp32 scale per tensor.  [LM-bus]
 * The kernels read a packed copy whose size is exactly the canonical size (9 bytes per 16 NVFP4
 * weights [SP-geom]; 1 byte per FP8 weight): 16-row blocks, each cut along K into chunks (256
 * weights wide for NVFP4, 128 for FP8) of two 8-row strips, stored row-block major so that one
 * row block's stream along K is contiguous and one chunk (2304 / 2048 bytes) is one bulk copy;
 * inside a strip the bytes follow the warp MMA's operand order (every thread's share of a 16-wide
 * k step is one aligned 16-byte read).
 * Requirements: N % 16 == 0; NVFP4 K % 256 == 0, FP8 K % 128 == 0; K <= 65536.  */

/* Packed size in bytes: N*K/16*9 (NVFP4) and N*K (FP8); 0 if N or K is unsupported. */
size_t vp_packed_bytes_nvfp4(int N, int K);
size_t vp_packed_bytes_fp8(int N, int K);

/* Device-to-device repack from the canonical layout.  codes: [N][K/2], scales: [N][K/16],
 * packed: vp_packed_bytes_nvfp4(N, K) bytes, all 16-byte aligned and not overlapping. */
vp_status vp_pack_nvfp4(const void* codes, const void* scales, int N, int K, void* packed,
                        size_t packed_bytes, void* stream);
/* w: [N][K] E4M3 bytes -> packed (vp_packed_bytes_fp8(N, K) bytes). */
vp_status vp_pack_fp8(const void* w, int N, int K, void* packed, size_t packed_bytes, void* stream);

/* Q4 (affine INT4, groups of 64 along K) [SP-q4]: codes [N][K/2] bytes, element 2j of a row is the
 * LOW nibble of byte j, an unsigned code q in 0..15; scales and biases [N][K/64] bf16;
 *   w[n][k] = scale[n][k/64] * q[n][k] + bias[n][k/64]
 * (the pages give the sizes, not the formula: the affine map is this library's reading).  Packed
 * size N*K/16*9 bytes, the canonical size; the packed layout has the NVFP4 geometry (256-wide
 * chunks, 1152-byte strips) with the codes in the order of an f16 magic-number conversion and each
 * row's four (scale, bias) pairs of a chunk in one 16-byte piece.  K % 256 == 0, N % 16 == 0.
 * codes and packed 16-byte aligned, scales and biases 2-byte aligned. */
size_t vp_packed_bytes_q4(int N, int K);
vp_status vp_pack_q4(const void* codes, const void* scales, const void* biases, int N, int K, void* packed,
                     size_t packed_bytes, void* stream);

/* ------------------------------------------------------------------ skinny linear layers
 *
 * y[m][n] = scale * sum_k x[m][k] * w[n][k], m < M, n < N, fp32 accumulation.  [LM-formats]
 *   NVFP4: w[n][k] = e2m1(code[n][k]) * e4m3(block_scale[n][k/16]); scale = the fp32 tensor
 *          scale (a multiplier).
 *   FP8:   w[n][k] = e4m3(w8[n][k]); scale = the fp32 per-tensor scale.
 * x: bf16 [M][K] row-major (device, 16-byte aligned); y: fp32 [M][N] row-major (device).
 * Shapes: 1 <= M <= 32, N % 16 == 0, K as for the packed layout, N*K < 2^40.
 * Work is split along K across warps and CTAs (split-K) with a fixed-order reduction, so results
 * are bit-identical from run to run.  [BS-ties] (split-K).  */
enum { VP_OP_NVFP4 = 0, VP_OP_FP8 = 1, VP_OP_HEAD = 2, VP_OP_ARGMAX = 3, VP_OP_Q4 = 4, VP_OP_SAMPLE = 5,
       VP_OP_ATTN = 6 };

/* Workspace bytes for one call of op (VP_OP_*) at the given shape; 0 if the shape is invalid. */
size_t vp_workspace_bytes(int op, int M, int N, int K);

vp_status vp_linear_nvfp4(const void* w_packed, float tensor_scale, const void* x, float* y, int M,
                          int N, int K, void* ws, size_t ws_bytes, void* stream);
vp_status vp_linear_fp8(const void* w_packed, float scale, const void* x, float* y, int M, int N,
                        int K, void* ws, size_t ws_bytes, void* stream);
/* Q4: y[m][n] = sum_k x[m][k] * (scale * q + bias)[n][k] [SP-q4].  Each 64-wide group is computed
 * as scale * (sum_k q x) + bias * (sum_k x): the codes enter the tensor core as exact f16 integers,
 * the group's activation sums come from the same tensor-core pass (a ones operand beside the codes),
 * and both terms are applied in fp32.  Workspace: vp_workspace_bytes(VP_OP_Q4, M, N, K).  Arguments, shapes and
 * errors otherwise as for vp_linear_nvfp4. */
vp_status vp_linear_q4(const void* w_packed, const void* x, float* y, int M, int N, int K, void* ws,
                       size_t ws_bytes, void* stream);

/* vp_linear_nvfp4 without a caller-provided workspace.  The pages describe no such call: it is
 * a convenience of this library for callers that cannot pass scratch memory -- a plugin or custom-
 * op interface whose fixed signature has no workspace argument, or a decode loop that must not
 * stall, where allocating device memory is not allowed (cudaMalloc / cudaFree synchronise the
 * device).  The call allocates nothing: it uses a fixed 8 MiB scratch array inside the library,
 * one per device, and computes exactly what vp_linear_nvfp4 computes (same kernel, same order of
 * reduction, so the same bits).
 *   - The first call on a device does the set-up (it looks up the scratch array's address, which
 *     may initialise the CUDA context); make it before any stream capture.
 *   - Every call clears the scratch's status word and counters on `stream` before its launch.
 *   - Shapes whose split-K bookkeeping needs more than the 8 MiB scratch (roughly: many rows times
 *     a K cut into several K slices, e.g. a 248320 x 5120 head at M = 32) return VP_ERR_WORKSPACE;
 *     use vp_linear_nvfp4 for them.
 *   - The scratch is shared by all calls on a device: calls that overlap in time (on different
 *     streams, or from different host threads) race and corrupt each other's results.  Order them
 *     on one stream.
 * Arguments, shapes and errors otherwise as for vp_linear_nvfp4. */
vp_status vp_linear_nvfp4_noalloc(const void* w_packed, float tensor_scale, const void* x, float* y, int M,
                                  int N, int K, void* stream);
/* The status word of the last vp_linear_nvfp4_noalloc call on this device (ordered on `stream`):
 * VP_OK, or VP_ERR_TIMEOUT when one of its bounded device waits gave up (its y is then not valid).
 * Copies the word to the host int *status and synchronises `stream`.  Each noalloc call clears the
 * word before its launch, so the status is that of the latest call enqueued before this one. */
vp_status vp_noalloc_read_status(int* status, void* stream);

/* ------------------------------------------------------------------ head + argmax + accept
 *
 * logits[m][v] = tensor_scale * sum_k x[m][k] * w[v][k] (NVFP4 head [V][K]), never materialised
 * unless `logits` is non-NULL; argmax[m] = the lowest index v with the largest logit (NaN counts
 * as -inf, -0 == +0) [BS-ties]; then per lane l (M = 8 * lanes, lanes 1..4) [LM-accept]:
 *   acc = 0; while (acc < 7 && argmax[8l + acc] == pending[8l + acc + 1]) acc++;
 *   n_commit[l] = acc + 1 (1..8);  committed[l][j] = argmax[8l + j] for j <= acc, -1 after.
 * pending[8l] is the lane's anchor (already committed) token and is not compared.
 * x: bf16 [M][K]; pending: int32 [M]; argmax: int32 [M]; n_commit: int32 [M/8];
 * committed: int32 [M/8][8]; logits: optional fp32 [M][V] (debug).  V % 16 == 0, K % 256 == 0. */
vp_status vp_head_argmax_accept(const void* w_packed, float tensor_scale, const void* x, int M,
                                int V, int K, const int32_t* pending, int32_t* argmax,
                                int32_t* n_commit, int32_t* committed, float* logits, void* ws,
                                size_t ws_bytes, void* stream);

/* The argmax + accept stage alone, over given fp32 logits [M][V] (any V >= 1; M = 8 * lanes).
 * It runs the same device reduction and acceptance code as vp_head_argmax_accept. */
vp_status vp_argmax_accept(const float* logits, int M, int V, const int32_t* pending,
                           int32_t* argmax, int32_t* n_commit, int32_t* committed, void* ws,
                           size_t ws_bytes, void* stream);
/* The same with R = rows verify rows per lane [WIDE] (1 <= rows <= 32, M = rows * lanes <= 128;
 * M > 32 only as runs of 32 rows, so M % 32 == 0 and 32 % rows == 0):
 *   acc = 0; while (acc < R - 1 && argmax[R l + acc] == pending[R l + acc + 1]) acc++;
 *   n_commit[l] = acc + 1 (1..R);  committed[l][j] = argmax[R l + j] for j <= acc, -1 after.
 * n_commit: int32 [M / R]; committed: int32 [M / R][R].  rows = 8 is vp_argmax_accept.  The
 * workspace is vp_workspace_bytes(VP_OP_ARGMAX, min(M, 32), V, 0) (runs of 32 rows reuse it, in
 * stream order).  VP_ERR_SHAPE for rows or M out of range, or M % rows != 0. */
vp_status vp_argmax_accept_rows(const float* logits, int M, int V, int rows, const int32_t* pending,
                                int32_t* argmax, int32_t* n_commit, int32_t* committed, void* ws,
                                size_t ws_bytes, void* stream);

/* Sampled acceptance over given fp32 logits [M][V] (M = 8 * lanes; 1 <= V <= 1,048,576)
 * [SP-sample].  Per row r, the target distribution p_r: the top_k (1..32, <= V) largest logits
 * (NaN as -inf; ties to the lower token index), p = exp((l - l_max) / temperature) normalised over
 * them, then the shortest prefix whose mass reaches top_p (0 < top_p <= 1), renormalised; every other
 * token has p = 0.  Per lane l, for draft j = 0..6 (d = pending[8l + j + 1], checked at row
 * r = 8l + j, q = the draft's probability of d):
 *   accept when uniforms[r][0] * q < p_r(d); otherwise draw the committed token from
 *   max(p_r - q_r, 0) (from p_r if that is zero everywhere) with uniforms[r][1] and stop;
 * when all 7 are accepted, draw the bonus token from p at row 8l + 7 with uniforms[8l + 7][1].
 * A draw with u over weights w in candidate order (larger logit first) takes the first i with
 * u * sum(w) < w_0 + .. + w_i.  The draft's distribution at row r is draft_tokens[r][0..15] /
 * draft_probs[r][0..15] (tokens not listed have q = 0); with both NULL each draft is a point mass
 * (q = 1 on d: a greedy drafter).  n_commit[l] = accepted + 1; committed[l] = the accepted drafts,
 * the drawn token, then -1.  uniforms: fp32 [M][2] in [0, 1), supplied by the caller (the library
 * draws no random numbers).  Arithmetic is fp32; decisions within rounding of a boundary may
 * differ from an fp64 evaluation.  One kernel launch.  Workspace: vp_workspace_bytes(VP_OP_SAMPLE,
 * M, V, 0), zero-filled once before its first use (its counters return to zero after each call).
 * Errors: VP_ERR_INVALID_ARG (null pointers, one of draft_tokens / draft_probs without the other,
 * temperature not finite and > 0, top_p outside (0, 1]), VP_ERR_SHAPE, VP_ERR_ALIGNMENT (4-byte
 * arrays, 256-byte workspace), VP_ERR_WORKSPACE. */
vp_status vp_sample_accept(const float* logits, int M, int V, float temperature, int top_k, float top_p,
                           const int32_t* pending, const int32_t* draft_tokens, const float* draft_probs,
                           const float* uniforms, int32_t* n_commit, int32_t* committed, void* ws,
                           size_t ws_bytes, void* stream);

/* Verify attention over a BF16 KV cache [LM-attn], for the attention layers' mixer core.  Lane l
 * (M = 8 * lanes) has ctx[l] cached positions in k_cache / v_cache [lanes][Hkv][cap][D]; the call
 * first writes the verify rows' keys / values k_new, v_new [M][Hkv][D] at positions ctx[l] + j
 * (j = 0..7), then for row r = 8l + j and q head h (kv head h / (Hq / Hkv)):
 *   out[r][h] = softmax_t(q[r][h] . k_t / sqrt(D)) over t = 0 .. ctx[l] + j, weighting v_t,
 *               times sigmoid(gate[r][h]) elementwise when gate is not NULL, rounded once to bf16.
 * q, gate, out: bf16 [M][Hq][D].  q and k are taken as given (after the layer's Q/K RMSNorm and RoPE,
 * which are elementwise steps before this one).  D = 256; Hq % Hkv == 0, Hq / Hkv <= 8; cap >= 8.
 * ctx is a device array [lanes] (so a device-resident loop can advance it); a lane with ctx[l] < 0 or
 * ctx[l] + 8 > cap is skipped (its output is zero and the workspace's status word reads
 * VP_ERR_SHAPE, see vp_read_status).  Partitions of at most 1,024 keys (shorter, in multiples of 64,
 * when that fills the GPU's 152 SMs in one wave) run in parallel (one CTA per partition, kv head and
 * lane) and are merged in a fixed order: bit-reproducible for a given cap.  QK^T runs on the
 * tensor core in bf16, P V in f16 (values must lie in f16's range, where bf16 values are exact).
 * Workspace: vp_workspace_bytes(VP_OP_ATTN, M, Hkv, cap), 256-byte aligned.  Three launches. */
vp_status vp_attention_verify(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                              const int32_t* ctx, int cap, const void* gate, void* out, int M, int Hq, int Hkv, int D,
                              void* ws, size_t ws_bytes, void* stream);

/* Gated DeltaNet verify scan [BS-gdn]: for lane l (M = 8 * lanes) and head h, from state_in
 * (fp32 [lanes][H][dv][dk], parity buffer A) over the lane's first rows[l] verify rows
 * (rows: device int32 [lanes], clamped to 0..8), the gated delta rule
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t
 * (the published Gated DeltaNet recurrence; the pages name the layer, not the formula), writing the
 * final state to state_out (parity buffer B; may equal state_in for an in-place update) and, when
 * out is not NULL, o_t to out (fp32 [M][H][dv], rows past rows[l] untouched).  q, k: bf16 [M][H][dk];
 * v: bf16 [M][H][dv]; alpha, beta: fp32 [M][H] (after the layer's gates; q, k, v after its short
 * convolution, activation and normalisation -- producer steps).  Verify: rows = 8 from A to B;
 * commit after a partial accept: rows = n_commit from A to B again -- the same kernel, so the
 * re-scan's state equals the verify scan's state after those rows bit for bit.  dk = dv = 128,
 * H 1..4096.
 * One launch, no workspace. */
vp_status vp_gdn_scan(const float* state_in, float* state_out, const void* q, const void* k, const void* v,
                      const float* alpha, const float* beta, const int32_t* rows, int M, int H, int dk, int dv,
                      float* out, void* stream);

/* ------------------------------------------------------------------ the verify pass
 *
 * The pass chains, for each layer l (attention when layer.kind == VP_LAYER_ATTN, else Gated
 * DeltaNet; the Splash geometry has every fourth layer attention [SP-geom]):
 *   r = RMSNorm(h)                                  (unit weight, eps; bf16 result)
 *   GDN:  u = FP8(in, r) [M][n_in];  z = bf16(u[:, :k_out]);  h = bf16(h + FP8(out, z))
 *   attn: q = FP8(q, r) [M][n_in], kv = FP8(kv, r) [M][n_kv] (streamed; unused by the stand-in
 *         mixer);  z = bf16(q[:, :k_out]);  h = bf16(h + FP8(o, z))
 *   r = RMSNorm(h);  a = bf16(silu(NVFP4(gate, r)) * NVFP4(up, r));  h = bf16(h + NVFP4(down, a))
 * and then r = RMSNorm(h); head + argmax + accept as vp_head_argmax_accept.
 * The mixer cores (Gated DeltaNet recurrence, attention over a KV cache) are outside the weight
 * stream and are replaced by the slice z = u[:, :k_out]; every weight GEMM of the pass
 * (17,555,292,160 bytes at the Qwen3.8-27B shapes [LM-bus]) is streamed.  */
enum { VP_LAYER_GDN = 0, VP_LAYER_ATTN = 1 };

typedef struct {
  int kind;          /* VP_LAYER_GDN or VP_LAYER_ATTN */
  const void* w_in;  /* FP8 packed [n_in][hidden]: GDN in-projection or attention q */
  float s_in;
  int n_in;
  const void* w_kv;  /* FP8 packed [n_kv][hidden] (attention only; NULL and 0 on GDN layers) */
  float s_kv;
  int n_kv;
  const void* w_out; /* FP8 packed [hidden][k_out]; k_out <= n_in */
  float s_out;
  int k_out;
  const void* w_gate; /* NVFP4 packed [inter][hidden] */
  float ts_gate;
  const void* w_up;   /* NVFP4 packed [inter][hidden] */
  float ts_up;
  const void* w_down; /* NVFP4 packed [hidden][inter] */
  float ts_down;
} vp_layer_desc;

typedef struct {
  const void* w; /* NVFP4 packed [vocab][hidden] */
  float ts;
  int vocab;
} vp_head_desc;

typedef struct vp_model vp_model;

/* Validates the descriptors (shapes as for the linear calls: hidden % 256 == 0, inter % 256 == 0,
 * k_out % 128 == 0, row counts % 16 == 0) and stores them with the pass's phase program (host
 * memory, owned by the model). */
vp_status vp_model_create(int hidden, int inter, float rms_eps, const vp_layer_desc* layers,
                          int n_layers, const vp_head_desc* head, vp_model** out);
void vp_model_destroy(vp_model* model);

/* Workspace bytes for vp_verify_pass (M = 8 * lanes) or vp_verify_blocks (M = 1..32) at M rows (0 if
 * invalid); for vp_verify_pass_rows also M = 64, 96, 128 (the workspace of 32 rows, which its passes
 * of 32 rows share). */
size_t vp_pass_workspace_bytes(const vp_model* model, int M);

/* One verify pass.  x0: bf16 [M][hidden] (the rows' input hidden states, read-only); pending,
 * argmax, n_commit, committed as for vp_head_argmax_accept; M = 8 * lanes, lanes 1..4.
 * trace: optional bf16 [2 * n_layers][M][hidden], the residual stream h after every mixer block
 * and every MLP block (debug; written by the residual epilogues).  logits: optional fp32
 * [M][vocab].  No host synchronisation, no allocation: capturable into a CUDA graph. */
vp_status vp_verify_pass(const vp_model* model, const void* x0, int M, const int32_t* pending,
                         int32_t* argmax, int32_t* n_commit, int32_t* committed, void* trace,
                         float* logits, void* ws, size_t ws_bytes, void* stream);
/* The verify pass with R = rows verify rows per lane [WIDE]: the same weight stream and logits for
 * the M rows (M = rows * lanes <= 32, 1 <= rows <= 32), the acceptance of vp_argmax_accept_rows in
 * the head (n_commit: int32 [M / R]; committed: int32 [M / R][R]).  One lane of 16 or 32 rows, or two
 * of 16, verify a deep lookup draft in one pass.  rows = 8 is vp_verify_pass; the workspace is
 * vp_pass_workspace_bytes(model, M).  M up to 128 (M % 32 == 0, 32 % rows == 0, trace NULL) runs as
 * M / 32 consecutive passes of 32 rows (whole lanes each) on the stream, sharing the workspace of
 * vp_pass_workspace_bytes(model, M) (= that of 32 rows): every pass streams the weights again. */
vp_status vp_verify_pass_rows(const vp_model* model, const void* x0, int M, int rows, const int32_t* pending,
                              int32_t* argmax, int32_t* n_commit, int32_t* committed, void* trace,
                              float* logits, void* ws, size_t ws_bytes, void* stream);

/* The verify pass with sampled instead of greedy acceptance [SP-sample]: the pass of
 * vp_verify_pass, whose head phase writes the fp32 logits [M][vocab] (into `logits` when non-NULL,
 * else into the workspace) and the argmax, then -- on the same stream, with no host in between -- the
 * sampled acceptance of vp_sample_accept over those logits (temperature, top_k, top_p, the drafts'
 * distributions draft_tokens / draft_probs or point masses when both are NULL, the caller's uniforms
 * [M][2]; see vp_sample_accept), which writes n_commit and committed.  argmax stays the greedy
 * target token of each row.  One launch more than vp_verify_pass and nothing read back to the host:
 * capturable into a CUDA graph.  Workspace: vp_pass_sampled_workspace_bytes(model, M) bytes,
 * zero-filled once.  Errors: as vp_verify_pass and vp_sample_accept (VP_ERR_SHAPE for a vocabulary
 * above 1,048,576 or top_k outside 1..min(32, vocab)). */
size_t vp_pass_sampled_workspace_bytes(const vp_model* model, int M);
vp_status vp_verify_pass_sampled(const vp_model* model, const void* x0, int M, const int32_t* pending,
                                 float temperature, int top_k, float top_p, const int32_t* draft_tokens,
                                 const float* draft_probs, const float* uniforms, int32_t* argmax,
                                 int32_t* n_commit, int32_t* committed, float* logits, void* ws,
                                 size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ the pass with the real mixer cores
 *
 * In place of the stand-in slice, each layer runs its own mixer core between its projections, all on
 * the device [LM-attn] [BS-gdn]:
 *   Gated DeltaNet: u = FP8(in, r) kept whole (rows: q (n_qk heads), k (n_qk), v (n_v), z (n_v), each
 *     d wide); a, b = r . A, r . B (BF16 [n_v][hidden] each, fp32 results); the causal depthwise
 *     4-tap convolution of u's q, k, v part over the lane's 3 earlier rows (window_a) and its 8 rows
 *     (tap 3 on the current row), SiLU; q, k over their per-head L2 norm (eps 1e-6 inside the root);
 *     q, k, v rounded to bf16, q / k head i serving v heads i * n_v / n_qk ..; alpha =
 *     exp(-exp(A_log) softplus(a + dt_bias)), beta = sigmoid(b); the gated delta rule of vp_gdn_scan
 *     from state_a into state_b over the 8 rows; bf16(o / sqrt(mean(o^2) + 1e-6) * norm_w * silu(z))
 *     per v head into the out-projection.
 *   attention: q + gate = FP8(q, r), k + v = FP8(kv, r), kept whole; q and k heads over their root
 *     mean square (eps 1e-6) times q_norm / k_norm, then the rotary embedding over the whole head at
 *     cache position ctx[lane] + j (base 10000), bf16; then vp_attention_verify (append k, v at ctx ..
 *     ctx + 7, causal softmax over the cache, times sigmoid(gate)) into the o-projection.
 * Rounding: bf16 at the projection outputs, the cores' inputs and outputs, and the residual.
 * State [BS-gdn]: the caller owns it (device memory, per layer).  The recurrent state is
 * double-buffered by step parity: a pass of parity p reads buffer p (0: state_a, 1: state_b) and writes
 * the other (the state after all 8 rows); it reads window_a and the cache rows before ctx, and writes
 * conv_hist (window_a's 3 rows then the 8 rows' conv inputs) and the cache rows ctx .. ctx + 7.  After
 * the acceptance, vp_commit_cores with the same parity re-scans each lane's n_commit rows from the
 * intact buffer p into the other one and rewrites window_a with rows n_commit .. n_commit + 2 of
 * conv_hist; the next pass then runs with parity 1 - p at ctx + n_commit.  d = 128 (the scan), D = 256
 * (the attention core), Hq / Hkv <= 8, ctx[lane] + 8 <= cap, hidden <= 8192. */
typedef struct {
  /* Gated DeltaNet layers */
  const void* w_a;       /* bf16 [n_v][hidden], 16-byte aligned */
  const void* w_b;       /* bf16 [n_v][hidden], 16-byte aligned */
  const void* conv_taps; /* bf16 [(2 n_qk + n_v) d][4] */
  const float* a_log;    /* fp32 [n_v] */
  const float* dt_bias;  /* fp32 [n_v] */
  const float* norm_w;   /* fp32 [d]: the gated RMSNorm's weight */
  float* state_a;        /* fp32 [lanes][n_v][d][d]: parity buffer A (read at parity 0, written at 1) */
  float* state_b;        /* fp32 [lanes][n_v][d][d]: parity buffer B (written at parity 0, read at 1) */
  void* window_a;        /* bf16 [lanes][3][(2 n_qk + n_v) d] (read by the pass, rewritten by the commit) */
  void* conv_hist;       /* bf16 [lanes][11][(2 n_qk + n_v) d] (written by the pass) */
  /* attention layers */
  const float* q_norm;   /* fp32 [D] */
  const float* k_norm;   /* fp32 [D] */
  void* k_cache;         /* bf16 [lanes][Hkv][cap][D] */
  void* v_cache;         /* bf16 [lanes][Hkv][cap][D] */
} vp_core_desc;

typedef struct {
  int n_qk, n_v, d;      /* Gated DeltaNet heads: q / k heads, v heads, head width */
  int Hq, Hkv, D, cap;   /* attention: query and key-value heads, head width, cache positions per lane */
} vp_core_geom;

/* Attaches the mixer cores to a model (one descriptor per layer; the model keeps the pointers).
 * Checks every layer's projection widths against the geometry: Gated DeltaNet n_in ==
 * (2 n_qk + 2 n_v) d and k_out == n_v d; attention n_in == 2 Hq D, n_kv == 2 Hkv D, k_out == Hq D
 * (VP_ERR_SHAPE); a missing pointer is VP_ERR_INVALID_ARG; w_a, w_b, the states and the caches not
 * 16-byte aligned (the other bf16 arrays not 2-byte aligned) is VP_ERR_ALIGNMENT. */
vp_status vp_model_set_cores(vp_model* model, const vp_core_geom* geom, const vp_core_desc* cores, int n_layers);
/* Workspace bytes of vp_verify_pass_cores at M rows (0 if the model has no cores or M is invalid). */
size_t vp_pass_cores_workspace_bytes(const vp_model* model, int M);
/* The verify pass with the real mixer cores (arguments as vp_verify_pass; ctx: device int32 [lanes],
 * the cached positions per lane; parity 0 or 1, see above, else VP_ERR_INVALID_ARG).  Launches: one
 * executor program per layer boundary and the cores' kernels in between, all on `stream`, nothing read
 * back to the host: capturable into a CUDA graph.  The workspace keeps each Gated DeltaNet layer's scan
 * inputs (q, k, v, alpha, beta of the 8 rows) for vp_commit_cores.  The attention core reports a lane
 * whose ctx + 8 exceeds cap in the workspace's status word (VP_ERR_SHAPE; that lane's cache is left as
 * it is). */
vp_status vp_verify_pass_cores(const vp_model* model, const void* x0, int M, const int32_t* ctx, int parity,
                               const int32_t* pending, int32_t* argmax, int32_t* n_commit, int32_t* committed,
                               void* trace, float* logits, void* ws, size_t ws_bytes, void* stream);
/* The commit of a pass of the given parity [BS-gdn]: for every Gated DeltaNet layer and lane, the
 * gated delta rule over the lane's first n_commit[lane] rows (device int32 [M / 8], clamped to 0..8)
 * from the intact parity buffer into the other, from the inputs the pass kept in `ws` (the same
 * arithmetic as the pass's scan: n_commit = 8 reproduces the pass's state bit for bit), and the next
 * window, rows n .. n + 2 of conv_hist, into window_a.  Run it after vp_verify_pass_cores on the same
 * stream and workspace, before the next pass.  One launch per 48 Gated DeltaNet layers; nothing read
 * back to the host.  Errors: VP_ERR_INVALID_ARG (no cores, NULL, parity), VP_ERR_SHAPE (M),
 * VP_ERR_ALIGNMENT, VP_ERR_WORKSPACE. */
vp_status vp_commit_cores(const vp_model* model, int M, const int32_t* n_commit, int parity, void* ws,
                          size_t ws_bytes, void* stream);

/* Kernel launches that vp_verify_pass_cores enqueues for a model with cores (0 without): one
 * executor program per segment (the first in-projection, then the 4 phases after each layer's
 * core, the last with the head), 1 per Gated DeltaNet core (A/B projections and gates, convolution
 * and norms, the scan and the gated norm in one launch of 4-CTA clusters) and 4 per attention core
 * (prep, cache append, partitions, merge), after one device-to-device copy of x0. */
int vp_pass_cores_launch_count(const vp_model* model);

/* Blocks [block_begin, block_end) of the pass on a caller-owned residual stream h (bf16
 * [M][hidden], M = 1..32: no acceptance runs, so M need not be whole lanes; updated in place); block
 * 2l is the mixer block of layer l and block 2l + 1 its MLP block, computed exactly as inside
 * vp_verify_pass (the same phases of the same kernel).
 * trace: optional bf16 [block_end - block_begin][M][hidden], h after each block.  Lets a
 * caller run part of the stream, or check one block against a reference from a known input. */
vp_status vp_verify_blocks(const vp_model* model, void* h, int M, int block_begin, int block_end, void* trace,
                           void* ws, size_t ws_bytes, void* stream);

/* Kernel launches that vp_verify_pass enqueues for a model (for launch accounting): the pass runs
 * as one persistent program of 4 phases per layer plus the head, at most 160 phases per launch,
 * after one device-to-device copy of x0. */
int vp_pass_launch_count(const vp_model* model);

/* The executor's phase timeline (no counterpart in the pages: a measurement aid).  Only a library
 * built with VP_PHASE_TRACE (libverify_trace.so) records it; any other build returns
 * VP_ERR_UNSUPPORTED.  Copies up to `bytes` of the timeline of the kernels that serve M rows into the
 * host buffer dst: uint64 [2][160][256][37], indexed [launch parity][phase of the launch][CTA][slot]
 * with globaltimer stamps in ns -- slot 0 phase start, 36 the staging's loads and row statistics
 * done, 1 end of the activation staging, 2 + w warp w done with its units, 18 + w warp w done with
 * the row blocks it shares within its CTA, 35 (K-sliced phases) the cross-slice sums done, 34 grid
 * barrier passed -- and the number of multi-phase launches completed so far into *launches (a
 * launch writes buffer launches % 2).
 * Synchronous (waits for the device). */
vp_status vp_trace_read(int M, void* dst, size_t bytes, unsigned* launches);

/* ------------------------------------------------------------------ device-resident decode loop [LOOP]
 *
 * Per lane l the decode state lives on the device: the token history hist[l][0 .. T_l) (int32
 * [lanes][cap], T_l = hist_len[l]; the last token is the anchor, already committed) and an optional
 * status word (set to VP_ERR_SHAPE by a kernel that met an out-of-range token or a full history; the
 * work it concerns is skipped).  Every call below is asynchronous on `stream`, synchronises nothing
 * and is CUDA-graph capturable. */

/* x[m][k] = bf16(e2m1(code) * e4m3(scale) * ts) of row tokens[m] of an NVFP4 table in the canonical
 * layout (codes [V][K/2], scales [V][K/16]), rounded once: the embedding gather.  x: bf16 [M][K].
 * K % 16 == 0, V * K < 2^40.  An out-of-range token gives a zero row and the status. */
vp_status vp_embed_nvfp4(const void* codes, const void* scales, float ts, const int32_t* tokens, int M, int V, int K,
                         void* x, int* status, void* stream);
/* Lookup drafts: pending[8l] = the anchor hist[l][T-1]; pending[8l + 1 + j] = hist[l][p + j] while
 * p + j < T, then the last copied token, where p (1 <= p < T) is the earlier position whose preceding
 * tokens match the history's last tokens for the most positions (at most max_match, at least one),
 * the latest p among equals; with no match every draft is the anchor.  lanes 1..4, cap < 2^24,
 * max_match 1..127; pending: int32 [8 lanes].  A lane with hist_len outside 1..cap gets all 8
 * pending entries 0, and the status. */
vp_status vp_lookup_drafts(const int32_t* hist, const int32_t* hist_len, int lanes, int cap, int max_match,
                           int32_t* pending, int* status, void* stream);
/* The same with R = rows entries per lane [WIDE]: pending[R l] = the anchor, then R - 1 drafts;
 * 1 <= rows <= 32, 1 <= lanes <= 32, lanes * rows <= 128; pending: int32 [R lanes].  rows = 8 is
 * vp_lookup_drafts. */
vp_status vp_lookup_drafts_rows(const int32_t* hist, const int32_t* hist_len, int lanes, int rows, int cap,
                                int max_match, int32_t* pending, int* status, void* stream);
/* Appends committed[l][0 .. n_commit[l]) to lane l's history (a lane that would overflow cap, or whose
 * n_commit is outside 1..8, is left as it is, with the status).  lanes 1..4; committed: int32
 * [lanes][8]. */
vp_status vp_commit_append(int32_t* hist, int32_t* hist_len, int lanes, int cap, const int32_t* n_commit,
                           const int32_t* committed, int* status, void* stream);
/* The same with committed rows of R = rows entries [WIDE] (n_commit outside 1..R: left as it is,
 * with the status); 1 <= rows <= 32, 1 <= lanes <= 32, lanes * rows <= 128; committed: int32
 * [lanes][R]. */
vp_status vp_commit_append_rows(int32_t* hist, int32_t* hist_len, int lanes, int rows, int cap,
                                const int32_t* n_commit, const int32_t* committed, int* status, void* stream);
/* `steps` rounds with no host in the loop: x0 = embed(pending) (the embedding table emb_codes /
 * emb_scales / emb_ts, [vocab][hidden]); vp_verify_pass; append the committed tokens; lookup drafts
 * into pending.  pending must hold the first round's anchor + drafts (e.g. from vp_lookup_drafts).
 * x0: bf16 [8 lanes][hidden]; argmax, n_commit, committed, ws as for vp_verify_pass (the last round's
 * values remain).  hidden must equal the model's hidden size (the embedding writes x0 rows of `hidden`
 * values and the pass reads rows of the model's width): VP_ERR_SHAPE otherwise.  All arguments are
 * checked before the first launch: a rejected call enqueues nothing (steps == 0: the checks alone). */
vp_status vp_decode_steps(const vp_model* model, int steps, const void* emb_codes, const void* emb_scales,
                          float emb_ts, int vocab, int hidden, int32_t* hist, int32_t* hist_len, int cap,
                          int lanes, int max_match, int32_t* pending, void* x0, int32_t* argmax, int32_t* n_commit,
                          int32_t* committed, void* ws, size_t ws_bytes, int* status, void* stream);
/* The decode loop with R = rows verify rows per lane [WIDE] (the pass, append and lookup of the
 * _rows calls above; 1 <= rows <= 32, lanes * rows <= 128, above 32 rows as vp_verify_pass_rows
 * takes them; x0: bf16 [R lanes][hidden]; pending, committed as there).  rows = 8 is
 * vp_decode_steps. */
vp_status vp_decode_steps_rows(const vp_model* model, int steps, int rows, const void* emb_codes,
                               const void* emb_scales, float emb_ts, int vocab, int hidden, int32_t* hist,
                               int32_t* hist_len, int cap, int lanes, int max_match, int32_t* pending, void* x0,
                               int32_t* argmax, int32_t* n_commit, int32_t* committed, void* ws, size_t ws_bytes,
                               int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_H_ */
