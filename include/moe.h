/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed int4 mixture-of-experts layer.
 *
 * The layer is the inference forward of a routed MoE block whose experts hold
 * PackedInt4Linear weights:
 *   - router: sigmoid affinities of fp32 logits plus an fp32 correction bias,
 *     top-k on the biased score, weights from the unbiased affinities divided
 *     by their sum + 1e-20 (Kimi K2.5 donor-reference page, equations
 *     "MoEGate.forward: logits", "Independent sigmoid scores for the router",
 *     "Bias the choice of experts while retaining original affinities",
 *     "Normalize the selected routing affinities");
 *   - dispatch: counts per expert, stable sort by expert, gather of token rows
 *     (Kimi K3 latent up-projection page, KimiSparseMoeBlock.moe_infer listing;
 *     donor-reference equations "DeepSeek MoE.moe_infer: tokens per expert" and
 *     "... sorted tokens"), done on the device with no host synchronisation;
 *   - experts: down(SiLU(gate(x)) * up(x)) with int4 weights (Kimi
 *     exact-generator adaptation page, sections "The proposed substitution",
 *     "The preserved forward form" and "Sources & provenance"; donor-reference
 *     equation "SwiGLU-style gated feed-forward projection");
 *   - combine: un-permute and fp32 sum of the k expert outputs times their
 *     routing weights (donor-reference equation "Sum the selected expert
 *     outputs with their routing weights"; moe_infer listing);
 *   - optional latent wrap: bf16 down-projection, RMSNorm, bf16
 *     up-projection (KimiSparseMoeBlock.forward listing, "Latent
 *     up-projection" section; donor-reference RMSNorm equations);
 *   - optional shared expert: a bf16 gated MLP on the full-width x added to
 *     the routed output (KimiSparseMoeBlock listing; donor-reference "Add an
 *     always-active shared expert");
 *   - weight preparation: bf16 weights to packed int4 with bf16 group-32
 *     scales (exact-generator page, "The proposed substitution").
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller unless the
 *     name says _host.  The library never allocates device memory in these
 *     calls; scratch space is the caller-provided workspace `ws` of
 *     `ws_bytes` bytes (256-byte aligned), sized by the matching
 *     *_workspace_size function.
 *   - bf16 tensors are passed as uint16_t bit patterns.  Every tensor is
 *     dense, row-major, with the shape given in brackets.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous and stream-ordered; they never synchronise the host, so a
 *     sequence of calls may be captured in a CUDA graph after one warm-up
 *     call per device (the warm-up loads the library's device code).
 *   - Packed int4 weights: int32 [E, N, K/8]; column 8*i + j of row n is
 *     nibble j (bits 4j..4j+3) of word i, a two's-complement value in
 *     [-8, 7].  Scales: bf16 [E, N, K/32], one per output row and 32-column
 *     group; W[n, c] = q[n, c] * scale[n, c / 32].
 *   - act_bits = 16: bf16 activations, weights dequantised exactly, fp32
 *     accumulation.  act_bits = 8 ("exact" mode): every int4 linear quantises
 *     its input per row to int8 (scale = max|v| / 127, q = clamp(rint(v /
 *     scale), -127, 127), IEEE fp32), integer products are summed exactly per
 *     32-column weight group, y = scale_x * sum_g scale_w[n, g] * P[g] in fp32.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code.  Argument errors are
 *     detected on the host before any launch.  Device-side problems are
 *     recorded in a per-device status word that moe_check_error() reads and
 *     clears: a bounded wait that ran out (MOE_ERR_TIMEOUT), offsets or row
 *     indices outside the stated capacity (MOE_ERR_INVALID), a value outside
 *     the range the kernels compute exactly (MOE_ERR_UNSUPPORTED).  The word
 *     keeps the first such error since the last check.  It is a report only:
 *     the kernels never read it, so an error recorded by one call does not
 *     change what later calls compute, whether or not anyone checks it.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID (-1)     /* null pointer, negative size, misaligned pointer */
#define MOE_ERR_UNSUPPORTED (-2) /* shape outside the supported set (see below) */
#define MOE_ERR_WORKSPACE (-3)   /* ws_bytes smaller than the *_workspace_size */
#define MOE_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed */
#define MOE_ERR_TIMEOUT (-5)     /* a device wait ran out (moe_check_error) */

/* Supported shapes: widths D, H, I multiples of 64; 1 <= k <= min(E, 32);
 * 1 <= E <= 2048; act_bits 16 or 8; T >= 0 (T = 0 is a no-op). */

typedef struct moe_config {
  int32_t T;        /* tokens */
  int32_t H;        /* width of x and of the output */
  int32_t E;        /* routed experts */
  int32_t k;        /* experts per token */
  int32_t I;        /* expert intermediate width */
  int32_t L;        /* latent width; 0 = no latent projections (experts see H) */
  int32_t act_bits; /* 16 or 8 */
  int32_t renorm;   /* 1: divide the top-k affinities by their sum + 1e-20 */
  float eps;        /* RMSNorm epsilon (latent path) */
  int32_t I_shared; /* shared-expert intermediate width; 0 = no shared expert */
} moe_config;

/* Weights of one layer.  D = L if L > 0 else H. */
typedef struct moe_weights {
  const float* router_w;       /* fp32 [E, H] */
  const float* router_bias;    /* fp32 [E] correction bias (ranking only) */
  const int32_t* gate_packed;  /* [E, I, D/8] */
  const uint16_t* gate_scale;  /* bf16 [E, I, D/32] */
  const int32_t* up_packed;    /* [E, I, D/8] */
  const uint16_t* up_scale;    /* bf16 [E, I, D/32] */
  const int32_t* down_packed;  /* [E, D, I/8] */
  const uint16_t* down_scale;  /* bf16 [E, D, I/32] */
  const uint16_t* lat_down;    /* bf16 [L, H]  (latent only) */
  const uint16_t* lat_norm;    /* bf16 [L] RMSNorm gain, NULL = no norm (latent only) */
  const uint16_t* lat_up;      /* bf16 [H, L]  (latent only) */
  const uint16_t* shared_gate; /* bf16 [I_shared, H]  (shared expert only) */
  const uint16_t* shared_up;   /* bf16 [I_shared, H] */
  const uint16_t* shared_down; /* bf16 [H, I_shared] */
  const uint16_t* router_w_terms; /* optional bf16 [3, E, H] from moe_router_prepare (used
                                     from T = 512 on), or NULL: split router_w on every call */
} moe_weights;

/* ---------------------------------------------------------------- router -- */

/* Workspace bytes of moe_route for T tokens, width H, E experts. */
size_t moe_route_workspace_size(int T, int H, int E);

/* Router (donor-reference equations "MoEGate.forward: logits" through
 * "Normalize the selected routing affinities").
 *   x         bf16 [T, H]
 *   w_router  fp32 [E, H];  bias fp32 [E]
 *   topk_idx  int32 [T, k] out: experts by descending s + b (equal scores:
 *             lower expert id first)
 *   topk_w    fp32 [T, k] out: s_j / (sum_j s_j + 1e-20) if renorm, else s_j
 * Logits are fp32 dot products of the bf16 x (exact in fp32) with w_router. */
int moe_route(const uint16_t* x, const float* w_router, const float* bias, int T, int H,
              int E, int k, int renorm, int32_t* topk_idx, float* topk_w, void* ws,
              size_t ws_bytes, void* stream);

/* One-time preparation of the router weight for calls of 512 tokens or more,
 * whose logits run on the tensor cores: w_terms (bf16 [3, E, H], 16-byte
 * aligned, caller-owned) receives three bf16 terms with
 * w_router = w_terms[0] + w_terms[1] + w_terms[2] (each term the bf16
 * rounding of what the previous ones leave), exactly for every weight w with
 * 2^-110 <= |w| < 3.38e38 and for zero (smaller weights leave remainders in
 * fp32's subnormal range); x times each term is exact in fp32.  Give it to moe_layer_forward in moe_weights.router_w_terms
 * (the same split is otherwise redone on every call).  Stream-ordered. */
int moe_router_prepare(const float* w_router, int E, int H, uint16_t* w_terms, void* stream);

/* -------------------------------------------------------------- dispatch -- */

size_t moe_dispatch_workspace_size(int T, int E, int k);

/* Count, stable sort and permute (moe_infer listing: one-hot counts, argsort,
 * gather), with no host synchronisation.
 *   topk_idx  int32 [T, k] (values in [0, E); each token lists an expert once)
 *   x         bf16 [T, D] rows the experts see
 *   counts    int32 [E] out: rows per expert (sum = T*k)
 *   offsets   int32 [E+1] out: exclusive prefix of counts
 *   row_token int32 [T*k] out: token of expert-sorted row r; rows of one
 *             expert are in ascending token order
 *   row_slot  int32 [T*k] out: top-k slot of row r
 *   inv_row   int32 [T*k] out: row of (token t, slot j) at index t*k + j
 *   x_sorted  out: bf16 [T*k, D] (act_bits 16) or int8 [T*k, D] (act_bits 8)
 *   x_scale   fp32 [T*k] out, act_bits 8 only (may be NULL for 16) */
int moe_dispatch(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E, int k,
                 int act_bits, int32_t* counts, int32_t* offsets, int32_t* row_token,
                 int32_t* row_slot, int32_t* inv_row, void* x_sorted, float* x_scale,
                 void* ws, size_t ws_bytes, void* stream);

/* Same as moe_dispatch, but x_sorted is written in the expert kernels' "pair
 * order": in every block of 8 columns the values are stored as columns
 * 0 4 1 5 2 6 3 7 (the order in which a packed int32 word pairs its
 * nibbles), as fp16 (act_bits 16; a bf16 value beyond the fp16 range records
 * MOE_ERR_UNSUPPORTED) or int8 (act_bits 8).  These are the rows
 * moe_expert_ffn_pairs reads; moe_layer_forward uses this pair of calls.
 * No page has this layout: it is the GB300 kernels' operand order. */
int moe_dispatch_pairs(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E, int k,
                       int act_bits, int32_t* counts, int32_t* offsets, int32_t* row_token,
                       int32_t* row_slot, int32_t* inv_row, void* x_sorted, float* x_scale,
                       void* ws, size_t ws_bytes, void* stream);

/* Same as moe_dispatch, for callers that cannot provide device memory.
 *
 * No page has a counterpart of this call: it exists for host programs that
 * cannot allocate device memory for a workspace -- for instance a plugin
 * whose host owns every device allocation and hands it only its input and
 * output buffers, or a runtime that forbids allocation once it is serving.
 * The call allocates nothing.  Its scratch (the per-chunk expert histograms
 * and in-chunk ranks) is one fixed 2 MiB array in the library's device data,
 * held on every GPU that loads the library until the process exits.
 *   Limit: ceil(T/32)*E rounded up to 64, plus T*k, must not exceed 524288
 *   (for example T = 16384 with E = 384, k = 8); larger requests return
 *   MOE_ERR_WORKSPACE before any launch.
 *   Each call looks up the array's device address in the current device's
 *   context (so the address stays right after a device reset); the first
 *   call on a device may load the library's device code, so make one call
 *   before any stream capture.
 *   All calls share the one array: calls whose executions overlap on the GPU
 *   (different streams, or several host threads) race and give wrong
 *   results.  Nothing in the array needs to start at zero.
 * Arguments, layouts, results and the other error codes are those of
 * moe_dispatch. */
int moe_dispatch_noalloc(const int32_t* topk_idx, const uint16_t* x, int T, int D, int E, int k,
                         int act_bits, int32_t* counts, int32_t* offsets, int32_t* row_token,
                         int32_t* row_slot, int32_t* inv_row, void* x_sorted, float* x_scale,
                         void* stream);

/* ------------------------------------------------------------ expert FFN -- */

size_t moe_expert_ffn_workspace_size(int E, int D, int I, int rows_max, int act_bits);

/* Gated expert MLP over expert-sorted rows (exact-generator adaptation page,
 * "The preserved forward form"): for rows r of expert e (offsets[e] <= r <
 * offsets[e+1]): y[r] = down_e( SiLU(gate_e(x[r])) * up_e(x[r]) ).
 *   x_sorted  bf16 or int8 [rows_max, D] (as written by moe_dispatch)
 *   x_scale   fp32 [rows_max] (act_bits 8 only)
 *   offsets   int32 [E+1], offsets[E] <= rows_max (checked on the device;
 *             a violation records MOE_ERR_INVALID and computes nothing)
 *   weights   gate/up [E, I, D/8] + bf16 [E, I, D/32]; down [E, D, I/8] +
 *             bf16 [E, D, I/32]
 *   y_sorted  bf16 [rows_max, D] out (rows >= offsets[E] untouched)
 * x_sorted is first copied into the kernels' pair order (see
 * moe_dispatch_pairs).  The intermediate h = SiLU(G) * U is computed in fp32
 * and stored as fp16 (bf16 in act_bits 8 mode, where it is re-quantised per
 * row before the down projection).  A value beyond the fp16 range records
 * MOE_ERR_UNSUPPORTED. */
int moe_expert_ffn(const void* x_sorted, const float* x_scale, const int32_t* offsets, int E,
                   int D, int I, int rows_max, const int32_t* gate_packed,
                   const uint16_t* gate_scale, const int32_t* up_packed, const uint16_t* up_scale,
                   const int32_t* down_packed, const uint16_t* down_scale, int act_bits,
                   uint16_t* y_sorted, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes of moe_expert_ffn_pairs (host only). */
size_t moe_expert_ffn_pairs_workspace_size(int E, int D, int I, int rows_max, int act_bits);

/* moe_expert_ffn over rows already in pair order, as moe_dispatch_pairs
 * writes them (fp16, or int8 with act_bits 8); same weights, offsets, y and
 * error behaviour, without the conversion pass of moe_expert_ffn.  The
 * intermediate h is kept in fp16 (act_bits 16). */
int moe_expert_ffn_pairs(const void* x_pairs, const float* x_scale, const int32_t* offsets, int E,
                         int D, int I, int rows_max, const int32_t* gate_packed,
                         const uint16_t* gate_scale, const int32_t* up_packed,
                         const uint16_t* up_scale, const int32_t* down_packed,
                         const uint16_t* down_scale, int act_bits, uint16_t* y_sorted, void* ws,
                         size_t ws_bytes, void* stream);

/* moe_expert_ffn_pairs for a caller that knows a bound on the rows of any one
 * expert: max_rows_per_expert >= the largest offsets[e+1] - offsets[e] (the
 * token count T of a layer call, as a token picks an expert at most once).
 * With a bound below 48 no tensor-core kernel is launched (the batch cannot
 * be prefill-shaped), and the CTA-pair kernels only when it reaches 129: the
 * launches that would find no work are skipped.  With a true bound the
 * results are the bits of moe_expert_ffn_pairs; a bound below the true
 * count can only move experts to the stream kernel (same values within
 * rounding, other bits), never leave one uncomputed.
 * max_rows_per_expert < 0: MOE_ERR_INVALID. */
int moe_expert_ffn_pairs_bounded(const void* x_pairs, const float* x_scale,
                                 const int32_t* offsets, int E, int D, int I, int rows_max,
                                 int max_rows_per_expert, const int32_t* gate_packed,
                                 const uint16_t* gate_scale, const int32_t* up_packed,
                                 const uint16_t* up_scale, const int32_t* down_packed,
                                 const uint16_t* down_scale, int act_bits, uint16_t* y_sorted,
                                 void* ws, size_t ws_bytes, void* stream);

/* The int16 / int64 reading of act_bits 16 for one grouped PackedInt4Linear
 * (exact-generator adaptation page, "Sources & provenance": PackedInt4Linear
 * with act_bits 16 by default and an "int64 exact int4 MAC"; the page does
 * not say what the 16 bits hold).  moe_int4_linear's act_bits 16 (and the
 * layer's) reads them as bf16 activations times exactly dequantised
 * weights; this call reads them as int16 codes with integer accumulation:
 *   per row, in IEEE fp32: a = max|x|; sx = a / 32767 (rounded to nearest);
 *   q = clamp(rint(x / sx), -32767, 32767), ties to even (a zero row: 0);
 *   per 32-column weight group g: P_g = sum q * q_w, an exact integer
 *   (|P_g| < 2^23; K * 8 * 32767 < 2^31, so K <= 8160);
 *   out[r][n] = sx * acc, acc = the fp32 chain fma(scale[n, g], P_g, acc)
 *   over the groups in K order from 0.
 *   x        bf16 [rows_max, K] (rows of expert e: offsets[e] .. offsets[e+1])
 *   offsets  int32 [E+1] (checked on the device: MOE_ERR_INVALID)
 *   w_packed int32 [E, N, K/8]; w_scale bf16 [E, N, K/32]
 *   out      fp32 [rows_max, N] (rows >= offsets[E] untouched)
 *   partials optional int32 [rows_max, N, K/32]: every P_g (NULL: none)
 * K % 32 == 0 and K <= 8160, else MOE_ERR_UNSUPPORTED.  SIMT integer
 * arithmetic (not a hot path of the layer). */
size_t moe_int4_linear_int16_workspace_size(int E, int K, int rows_max);
int moe_int4_linear_int16(const uint16_t* x, const int32_t* offsets, int E, int K, int N,
                          int rows_max, const int32_t* w_packed, const uint16_t* w_scale,
                          float* out, int32_t* partials, void* ws, size_t ws_bytes, void* stream);

/* The int16 codes of that reading on their own: v bf16 [R, C] -> q int16
 * [R, C], scale fp32 [R] (the steps above). */
int moe_quantize_rows_int16(const uint16_t* v, int R, int C, int16_t* q, float* scale,
                            void* stream);

/* Workspace bytes of moe_int4_linear (host only). */
size_t moe_int4_linear_workspace_size(int E, int K, int rows_max);

/* One grouped PackedInt4Linear (exact-generator adaptation page, "Sources &
 * provenance"): out[r] = x[r] W_e^T for the rows r of expert e, fp32 out.
 *   x         bf16 or int8 [rows_max, K]; x_scale fp32 [rows_max] (act_bits 8)
 *   w_packed  int32 [E, N, K/8]; w_scale bf16 [E, N, K/32]
 *   out       fp32 [rows_max, N], 16-byte aligned
 * When an expert has at least 48 rows and K % 64 == 0, every expert runs on
 * the tensor-core kernels (with act_bits 16 the large experts on the
 * CTA-pair kernel, see moe_set_tc_pair), otherwise every expert on the
 * stream kernel (the
 * choice is taken on the device from the offsets).  With
 * act_bits 8 both kernels form the exact integer partial P_g of every
 * 32-column weight group and give the same bits: y = x_scale * acc, acc the
 * fp32 chain fma(scale[n, g], P_g, acc) over the groups in K order. */
int moe_int4_linear(const void* x, const float* x_scale, const int32_t* offsets, int E, int K,
                    int N, int rows_max, const int32_t* w_packed, const uint16_t* w_scale,
                    int act_bits, float* out, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes of moe_int4_linear_partials (host only). */
size_t moe_int4_linear_partials_workspace_size(int E, int K, int rows_max);

/* For tests: the exact-mode integer accumulators of one grouped
 * PackedInt4Linear (exact-generator adaptation page, "Sources & provenance":
 * the exact int4 multiply-accumulate; "The preserved forward form":
 * accumulator bounds).  Runs moe_int4_linear's act_bits 8 computation for
 * every expert on the kernel `kernel` names -- 0: the stream kernel (chunks
 * of <= 16 rows), 1: the tensor-core kernel (chunks of <= 128 rows) --
 * whatever the row counts, and also stores the integer partial of every
 * 32-column weight group:
 *   partials  int32 [rows_max, N, K/32] out:
 *             P[r, n, g] = sum_{c in group g} x[r, c] * q_w[n, c], exact
 *             (|P| <= 32 * 8 * 127);
 *   out       fp32 [rows_max, N] out: y[r, n] = x_scale[r] * acc, acc the
 *             fp32 chain acc = fma(scale[n, g], P[r, n, g], acc) over g in
 *             K order from 0 -- the bits moe_int4_linear gives on either
 *             kernel.
 * x int8 [rows_max, K] (16-byte aligned), x_scale fp32 [rows_max]; weights,
 * offsets, K % 64 == 0 and the error codes as moe_int4_linear.  Rows
 * outside every expert are left untouched. */
int moe_int4_linear_partials(const int8_t* x, const float* x_scale, const int32_t* offsets, int E,
                             int K, int N, int rows_max, const int32_t* w_packed,
                             const uint16_t* w_scale, int kernel, float* out, int32_t* partials,
                             void* ws, size_t ws_bytes, void* stream);

/* Per-row symmetric int8 quantisation (the act_bits 8 input step):
 * v bf16 [R, C] -> q int8 [R, C], scale fp32 [R].  R rows, C % 64 == 0. */
int moe_quantize_rows(const uint16_t* v, int R, int C, int8_t* q, float* scale, void* stream);

/* int4 weight quantiser (the conversion the "Kimi exact-generator adaptation"
 * page names in section "The proposed substitution": ExactLinear.from_weight
 * with a four-bit choice and group size 32; the page gives no rounding rule).
 * Reading, per row and 32-column group, in IEEE float32: a = max|w|;
 * s = bf16(a / 7) (division rounded to nearest, then to bf16, ties to even);
 * q = clamp(rint(w / s), -8, 7) with the stored s, ties to even; s = 0 gives
 * q = 0.
 *   w       bf16 [N, K] row-major, device, 16-byte aligned (stacked experts
 *           [E, N, K] are rows E*N);
 *   packed  int32 [N, K/8] out, device, 16-byte aligned: nibble j (bits
 *           4j..4j+3) of word i is column 8i+j, two's complement;
 *   scale   bf16 [N, K/32] out, device.
 * K % 32 == 0 (else MOE_ERR_UNSUPPORTED).  A non-finite weight records
 * MOE_ERR_UNSUPPORTED in the device status word (moe_check_error); its group
 * gets s = 0.  Caller-owned buffers; stream-ordered, no host sync. */
int moe_quantize_int4(const uint16_t* w, int N, int K, int32_t* packed, uint16_t* scale,
                      void* stream);

/* 8-bit weight quantiser: the eight-bit choice of the same conversion
 * (ExactLinear.from_weight with "four-bit or eight-bit choices and a group
 * size of 32", "Kimi exact-generator adaptation" page, section "The proposed
 * substitution"; no rounding rule is given).  Reading, per row and 32-column
 * group, in IEEE float32: a = max|w|; s = bf16(a / 127) (division rounded to
 * nearest, then to bf16, ties to even); q = clamp(rint(w / s), -127, 127)
 * with the stored s, ties to even; s = 0 gives q = 0.
 *   w      bf16 [N, K] row-major, device, 16-byte aligned;
 *   q      int8 [N, K] out, device, 16-byte aligned, column order;
 *   scale  bf16 [N, K/32] out, device.
 * K % 32 == 0 (else MOE_ERR_UNSUPPORTED).  A non-finite weight records
 * MOE_ERR_UNSUPPORTED in the device status word; its group gets s = 0.
 * Caller-owned buffers; stream-ordered, no host sync. */
int moe_quantize_int8(const uint16_t* w, int N, int K, int8_t* q, uint16_t* scale, void* stream);

/* --------------------------------------------------------------- combine -- */

/* Un-permute and weighted sum (moe_infer listing; donor-reference "Sum the
 * selected expert outputs with their routing weights"):
 *   out[t] = bf16( sum_j fp32(y_sorted[inv_row[t*k + j]]) * topk_w[t*k + j] ),
 * j ascending.  y_sorted bf16 [T*k, D], inv_row int32 [T*k], topk_w fp32
 * [T*k], out bf16 [T, D].  A row index outside [0, T*k) is skipped (the slot
 * adds nothing) and records MOE_ERR_INVALID. */
int moe_combine(const uint16_t* y_sorted, const int32_t* inv_row, const float* topk_w, int T,
                int D, int k, uint16_t* out, void* stream);

/* ---------------------------------------------------------------- latent -- */

/* y = x W^T with bf16 operands, fp32 accumulation, bf16 out ([out, in]
 * weight layout, "Latent up-projection" section).  x [M, K], w [N, K],
 * y [M, N]; K % 32 == 0. */
int moe_linear_bf16(const uint16_t* x, const uint16_t* w, int M, int N, int K, uint16_t* y,
                    void* stream);

/* y = bf16( x / sqrt(mean(x^2) + eps) * gain ) per row, fp32 arithmetic
 * (donor-reference RMSNorm equations).  x, y bf16 [M, N]; gain bf16 [N]. */
int moe_rmsnorm(const uint16_t* x, const uint16_t* gain, int M, int N, float eps, uint16_t* y,
                void* stream);

/* --------------------------------------------------------- shared expert -- */

/* Workspace bytes of moe_shared_expert. */
size_t moe_shared_expert_workspace_size(int T, int H, int I);

/* The always-active shared expert, added to an output ("Kimi K3 latent
 * up-projection" page, KimiSparseMoeBlock listing: shared_experts = KimiMLP
 * of moe_intermediate_size * num_shared_experts features and
 * y = y + shared_experts(identity); "Kimi K2.5 donor reference" page, "Add an
 * always-active shared expert"; the exact-generator page keeps shared experts
 * as ordinary bf16 linear modules):
 *   out = bf16( (accumulate ? out : 0) + down( bf16(SiLU(gate(x)) * up(x)) ) )
 * with fp32 accumulation of every product and h stored in bf16.
 *   x       bf16 [T, H] (the full-width layer input), 16-byte aligned
 *   gate_w, up_w  bf16 [I, H];  down_w bf16 [H, I]  (nn.Linear [out, in])
 *   out     bf16 [T, H], read when accumulate != 0, written
 * H % 64 == 0 and I % 64 == 0 (else MOE_ERR_UNSUPPORTED).  Caller-owned
 * device buffers and workspace (256-byte aligned); stream-ordered. */
int moe_shared_expert(const uint16_t* x, int T, int H, int I, const uint16_t* gate_w,
                      const uint16_t* up_w, const uint16_t* down_w, int accumulate, uint16_t* out,
                      void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------- layer -- */

/* Workspace bytes of moe_layer_forward / moe_layer_forward_host. */
size_t moe_workspace_size(const moe_config* cfg);

/* The whole layer (KimiSparseMoeBlock.forward listing): route on x, optional
 * latent down-projection, dispatch, experts, combine (+ RMSNorm and
 * up-projection when cfg->L > 0), then, when cfg->I_shared > 0, the shared
 * expert on x added to the routed output (summed in fp32, one bf16 rounding).
 *   x bf16 [T, H] in, out bf16 [T, H] out.  All intermediates live in ws. */
int moe_layer_forward(const moe_config* cfg, const moe_weights* w, const uint16_t* x,
                      uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* Same, with x and out in HOST memory (pinned memory gives asynchronous
 * copies): copies x to the device, runs the layer and copies out back, all
 * on `stream`.  The caller synchronises the stream before reading out_host. */
int moe_layer_forward_host(const moe_config* cfg, const moe_weights* w, const uint16_t* x_host,
                           uint16_t* out_host, void* ws, size_t ws_bytes, void* stream);

/* A captured layer call: one moe_layer_forward (host == 0) or
 * moe_layer_forward_host (host != 0) call with exactly these arguments,
 * recorded once as a CUDA graph, for callers that run the layer again and
 * again on the same buffers (a serving loop).  No page has this call: it
 * replaces the per-call launches of the library's kernels (8 to 18 per layer
 * in the measured workloads) with one graph launch.  All pointers are baked in: the weights, x,
 * out (pinned host memory when host != 0) and ws must stay valid and are
 * re-read on every launch.  The capture runs on `stream`, which must not be
 * capturing already, in thread-local mode; nothing executes during it.
 * Argument errors are those of the captured call, returned before any
 * capture; *graph is NULL on every error. */
typedef struct moe_layer_graph moe_layer_graph;
int moe_layer_graph_create(const moe_config* cfg, const moe_weights* w, const void* x, void* out,
                           int host, void* ws, size_t ws_bytes, void* stream,
                           moe_layer_graph** graph);

/* Runs the captured call on `stream` (stream-ordered, no host sync): the
 * same kernels, results and device status behaviour as the call it captured.
 * moe_launch_count() advances by the captured kernel count. */
int moe_layer_graph_launch(const moe_layer_graph* graph, void* stream);

/* Frees a captured call (NULL is ignored); launches already issued finish. */
void moe_layer_graph_destroy(moe_layer_graph* graph);

/* Pipelined layer calls on host buffers, for a serving loop that feeds one
 * call after another from pinned host memory (no page has this call).  Call n
 * of a pipe copies its x_host in on a stream of the pipe, runs the layer as a
 * captured graph (moe_layer_graph) on `stream` in device slot n % 2, and
 * copies out back on a second stream of the pipe, so that the copies of one
 * call overlap the compute of the calls before and after it.  The results
 * are those of moe_layer_forward_host.
 *   moe_layer_pipe_workspace_size: ws bytes (the layer's workspace plus two
 *     device slots for x and out; 0 for an invalid cfg).
 *   moe_layer_pipe_create: checks the arguments (those of moe_layer_forward,
 *     T > 0), creates the pipe's two streams and events and captures the two
 *     slots' graphs on `stream`, which must not be capturing.  The arrays w
 *     points to and ws must stay valid until destroy.  *pipe is NULL on
 *     every error.
 *   moe_layer_pipe_submit: enqueues one call (no host sync); x_host and
 *     out_host (T x H bf16, pinned) must stay valid until the call's output
 *     copy has finished; every submit to a pipe uses the same `stream`.
 *   moe_layer_pipe_join: makes `stream` wait for the output copies of every
 *     call submitted so far (synchronise the stream before reading them).
 *   moe_layer_pipe_destroy: waits for the pipe's copies, then frees it
 *     (NULL is ignored). */
typedef struct moe_layer_pipe moe_layer_pipe;
size_t moe_layer_pipe_workspace_size(const moe_config* cfg);
int moe_layer_pipe_create(const moe_config* cfg, const moe_weights* w, void* ws, size_t ws_bytes,
                          void* stream, moe_layer_pipe** pipe);
int moe_layer_pipe_submit(moe_layer_pipe* pipe, const uint16_t* x_host, uint16_t* out_host,
                          void* stream);
int moe_layer_pipe_join(moe_layer_pipe* pipe, void* stream);
void moe_layer_pipe_destroy(moe_layer_pipe* pipe);

/* ------------------------------------------------------------ status etc -- */

/* Synchronises `stream`, then returns and clears the current device's
 * status word: MOE_OK, or the first of MOE_ERR_TIMEOUT, MOE_ERR_INVALID and
 * MOE_ERR_UNSUPPORTED recorded on the device since the last check (see the
 * conventions above).  Returns MOE_ERR_CUDA if the stream reports a CUDA
 * error.  It blocks the host, so a serving loop calls it off the hot path
 * (for instance once per batch of steps); not checking is harmless, since
 * no kernel reads the word. */
int moe_check_error(void* stream);

/* Launches a kernel that waits on a barrier nothing completes, with a limit
 * of `limit_ns` nanoseconds (1e3 .. 5e9).  When the limit runs out the kernel
 * records MOE_ERR_TIMEOUT and returns; moe_check_error() then reports it.
 * Exercises the bounded-wait path of the pipelined kernels. */
int moe_wait_selftest(int64_t limit_ns, void* stream);

/* For tests: the exit paths of the pipelined expert kernels.  Runs
 * moe_int4_linear (same arguments, workspace of
 * moe_int4_linear_workspace_size) on the kernel `kernel` names -- 0: the
 * stream kernel (chunks of <= 16 rows), 1: the tensor-core kernel (the
 * act_bits 16 one, or the exact one for act_bits 8; chunks of <= 128 rows),
 * 2: the CTA-pair tensor-core kernel (act_bits 16 only, chunks of <= 256
 * rows; MOE_ERR_UNSUPPORTED where no cluster of two fits), 3: the small-tile
 * layout of the act_bits 16 tensor-core kernel (chunks of <= 64 rows)
 * -- in a build of it whose producer stops before its copy stage
 * `stall_stage` (counted per CTA from 0), as if those copies never arrived,
 * with every bounded wait limited to `limit_ns` (1e3 .. 5e9).  The other
 * roles' waits then run out: the kernel records MOE_ERR_TIMEOUT, lets every
 * copy and MMA it issued complete, frees its tensor memory and returns;
 * moe_check_error() reports the time-out and later calls run normally.  The
 * production kernels do not contain the stop. */
int moe_int4_linear_stall_selftest(const void* x, const float* x_scale, const int32_t* offsets,
                                   int E, int K, int N, int rows_max, const int32_t* w_packed,
                                   const uint16_t* w_scale, int act_bits, int kernel,
                                   int stall_stage, int64_t limit_ns, float* out, void* ws,
                                   size_t ws_bytes, void* stream);

/* Which tensor-core kernels run the act_bits 16 expert GEMMs of
 * moe_expert_ffn, moe_layer_forward and moe_int4_linear for prefill-shaped
 * batches.  enable != 0 (the default), where a cluster of two CTAs fits on
 * the device: the experts with at least 129 rows run on the CTA-pair kernels
 * -- clusters of two CTAs whose MMAs (tcgen05 cta_group::2) take 256 weight
 * rows over two SMs, on chunks of up to 256 token rows -- and the others on
 * the one-CTA kernels (128 weight rows per MMA, chunks of up to 128 rows; for
 * experts of at most 64 rows a layout with 64-row tiles and deeper rings);
 * the pair kernels are launched only when the batch's mean expert load
 * rows_max / E is at least 64 rows.  enable == 0: every expert on the one-CTA
 * kernels.  Both kernels take the same K steps of 16 columns for every output
 * and give the same bits (a GPU test checks it).  Process-wide, host only;
 * returns the previous setting.  For tests and measurements that compare the
 * two. */
int moe_set_tc_pair(int enable);

/* Human-readable name of a status code. */
const char* moe_status_string(int status);

/* Name of the CUDA runtime error (e.g. "cudaErrorInvalidValue") that last
 * made a call of this library return MOE_ERR_CUDA on the calling thread, or
 * "cudaSuccess" when none has.  A MOE_ERR_CUDA from a failed tensor-map
 * encoding (a driver call) records no runtime error.  Host only; never
 * synchronises; the returned string is static. */
const char* moe_last_cuda_error(void);

/* Library version string. */
const char* moe_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads), counted on the host as each launch is issued; a launch that
 * fails to start is counted too.  For measurement: the difference of two reads
 * around a region is the number of kernels of the library issued in it. */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
