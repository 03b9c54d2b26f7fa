/*
 * fme.h -- C ABI of libfme.so: the routed-expert MoE decode layer (FP8 and
 * NVFP4) and the FP8 shared expert, as hand-written sm_103a CUDA kernels.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named x, logits, bias, w13, s13, w2, s2, topk_ids, topk_weights,
 *   packed (inputs) and out, ids, weights, y, gate_up, dst (outputs) are
 *   DEVICE pointers; the caller owns every buffer. The library never
 *   allocates, frees or caches device memory.
 * - Matrices are dense row-major (last index fastest). Every device pointer
 *   must be 16-byte aligned.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream). Calls are asynchronous on it and never synchronise the host.
 * - Return value: FME_OK, or a negative fme_status when the host-side checks
 *   reject the arguments or the launch fails. fme_last_error() then holds a
 *   one-line reason (thread-local). Device-side faults of the bounded waits
 *   are reported through the workspace error word (fme_workspace_error).
 * - Workspace: caller-owned device scratch of at least the size the matching
 *   *_workspace() function returns. It must be zero-filled before its first
 *   use (fme_workspace_clear). Every successful call leaves its counters at
 *   zero again, so one workspace serves any number of calls issued in stream
 *   order, including calls with fewer tokens M than it was sized for (same
 *   other sizes). fme_moe_routed_fp8 and fme_moe_layer_fp8 calls with the same
 *   H, I, E and top_k may share one workspace (sized for the larger need);
 *   the shared-expert and NVFP4 calls each need their own. Two calls that
 *   overlap on the GPU need two workspaces. After a device-side error, clear
 *   it again before reuse.
 * - BF16 is IEEE bfloat16 (uint16 bit patterns). FP8 is E4M3 ("e4m3fn": no
 *   infinities, 0x7F/0xFF are NaN). FP4 is E2M1, sign in bit 3.
 */
#ifndef FME_H_
#define FME_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FME_OK = 0,
  FME_EINVAL = -1,       /* bad shape, count or null pointer */
  FME_EUNSUPPORTED = -2, /* valid request outside the supported shape range */
  FME_EALIGN = -3,       /* a pointer is not 16-byte aligned */
  FME_ECUDA = -4,        /* a CUDA runtime call failed (message has the name) */
  FME_ETIMEOUT = -5,     /* a device-side bounded wait gave up */
  FME_EWORKSPACE = -6    /* workspace missing or too small */
} fme_status;

typedef enum { FME_F32 = 0, FME_BF16 = 1 } fme_dtype;

/* One-line reason for the last non-OK status returned on this host thread. */
const char* fme_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int fme_version(void);

/*
 * Routed FP8 MoE layer for M decode tokens.
 *
 * Source: "vllm.models.glm5next.nvidia.specialized_decode.mega_moe",
 * MegaExperts.__call__ and _MegaKernel (top_k_pick, the epilogue x-quant,
 * GEMM1 and GEMM2 epilogues, hidden_block). Per token t and pick r:
 *   routing  s = sigmoid(logits[t]); key = s + bias; the top_k largest keys
 *            (ties: lower expert) in descending key order -> ids[t, r];
 *            weights[t, r] = s_r / (float sum of picked s) * scale (bias is
 *            used for selection only).
 *   x-quant  per 128-block of x[t]: sx = max(amax, 1e-10) / 448 (rounded up to
 *            a power of two when ue8m0), q = e4m3(x * (1 / sx)).
 *   GEMM1    y[n] = sum_b (sum_{k in b} W13[e, n, k] q[k]) * (s13[e, n/128, b] * sx[b]),
 *            n < 2I; rows [0, I) are "up", rows [I, 2I) are "gate".
 *   SwiGLU   h = silu(min(gate, limit)) * clamp(up, -limit, limit).
 *   h-quant  per 128-block of h: sh = max(amax, 1e-10) / 448 (power of two when
 *            ue8m0), qh = e4m3(h / sh).
 *   GEMM2    out[t*top_k + r, m] = bf16(sum_b (sum_j W2[e, m, j] qh[j]) * (s2[e, m/128, b] * sh[b])).
 * The route rows are NOT multiplied by the routing weights.
 *
 * Arguments:
 *   x       [M, H] BF16 tokens.
 *   logits  [M, E] router logits, dtype logits_dtype (FME_F32 or FME_BF16).
 *   bias    [E] FP32 score-correction bias.
 *   w13     [E, 2I, H] E4M3 (up rows, then gate rows); s13 [E, 2I/128, H/128] FP32.
 *   w2      [E, H, I] E4M3; s2 [E, H/128, I/128] FP32.
 *   M in [1, 64], H and I multiples of 128 with H, I <= 8192, E in [1, 1024],
 *   top_k in [1, min(E, 32)], limit > 0 (+inf allowed), scale finite.
 *   out     [M*top_k, H] BF16 (row t*top_k + r), ids [M, top_k] int32,
 *   weights [M, top_k] FP32.
 *   workspace / workspace_bytes: see fme_moe_routed_fp8_workspace.
 * Each touched expert's weights are read from HBM once per call, whatever
 * the number of routes that picked it.
 */
int fme_moe_routed_fp8(const void* x, const void* logits, int logits_dtype, const float* bias,
                       const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                       int M, int H, int I, int E, int top_k, float limit, float scale, int ue8m0,
                       void* out, int32_t* ids, float* weights, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Workspace bytes fme_moe_routed_fp8 needs for these sizes (0 on bad sizes). */
size_t fme_moe_routed_fp8_workspace(int M, int H, int I, int E, int top_k);

/*
 * fme_moe_routed_fp8 with MXFP8 activations: x arrives as E4M3 values with one
 * E8M0 scale per 32 values (the format of the expert-parallel dispatch,
 * fme_mxfp8_quantize), so GEMM1 skips the per-128 quantisation of x.
 *
 * Sources: the routed layer as fme_moe_routed_fp8 ("mega_moe"); the
 * activation format from "vllm.models.kimi_k3.nvidia.specialized_decode.
 * cutedsl.moe.ep.comm" (EpDispatch). The pages do not print this product; it
 * is y[n] = sum over K blocks b and their 32-value blocks s of
 * P[n, b, s] * (w_scale[n/128, b] * 2^(e[b, s] - 127)), each P the FP32
 * partial sum of one 32-value block (its own accumulator column), the
 * scaled partials summed in FP32. GEMM2 and everything after it as
 * fme_moe_routed_fp8.
 *
 * Arguments: xq [M, H] E4M3 bytes and xscales [M, H/32] E8M0 bytes in place
 * of x; the rest as fme_moe_routed_fp8 (same workspace size function; the two
 * entries may share a workspace). Every pointer 16-byte aligned except
 * xscales. Errors as fme_moe_routed_fp8.
 */
int fme_moe_routed_fp8_mx(const uint8_t* xq, const uint8_t* xscales, const void* logits, int logits_dtype,
                          const float* bias, const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                          int M, int H, int I, int E, int top_k, float limit, float scale, int ue8m0, void* out,
                          int32_t* ids, float* weights, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fme_moe_routed_fp8 for callers that cannot allocate device memory.
 *
 * No counterpart in the pages: this is a library convenience. Some callers
 * cannot call cudaMalloc (code running inside another owner's memory pool, a
 * plug-in whose host forbids device allocations after start-up, paths that
 * run while a graph is being captured), so they cannot hand over a workspace.
 * This variant takes the same arguments minus the workspace and uses an
 * 64 MiB scratch array compiled into libfme.so instead. A GPU holds that
 * array from the moment the module that defines it is loaded there (with
 * CUDA's default lazy loading, the variant's first call on that GPU) until
 * the process exits. It allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * - Size limit: the call must need at most 64 MiB of workspace
 *   (fme_moe_routed_fp8_workspace <= 67108864; e.g. the DeepSeek-V3 shape
 *   H = 7168, I = 2048, top_k = 8 up to M = 63 tokens). Larger requests
 *   return FME_EUNSUPPORTED.
 * - First call per device: it looks up the array's device address with that
 *   device current. Make that first call before any stream capture. The
 *   address is cached per device and looked up again when the device's
 *   context has changed (after cudaDeviceReset).
 * - Every call shares the one array and zeroes its counters first, so calls
 *   that overlap on the GPU (other streams, other host threads) race and
 *   corrupt each other: issue them in one stream order.
 * - Arguments are checked exactly as fme_moe_routed_fp8 checks them, before
 *   the array is touched: a rejected call leaves it as it was.
 * - The device error word lives in the shared array. Calls do not clear it:
 *   a bit set by any call stays set until fme_moe_routed_fp8_noalloc_error
 *   reads it.
 */
int fme_moe_routed_fp8_noalloc(const void* x, const void* logits, int logits_dtype, const float* bias,
                               const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                               int M, int H, int I, int E, int top_k, float limit, float scale, int ue8m0,
                               void* out, int32_t* ids, float* weights, void* stream);

/*
 * Read and clear the device error word of fme_moe_routed_fp8_noalloc on the
 * current device (synchronises stream). No counterpart in the pages. The
 * bits are those of fme_workspace_error and accumulate over every no-alloc
 * call since the last read. Allocates nothing. *code receives the word;
 * returns FME_ETIMEOUT when it is non-zero, FME_OK otherwise.
 */
int fme_moe_routed_fp8_noalloc_error(int* code, void* stream);

/*
 * FP8 shared expert for M decode tokens.
 *
 * Source: "vllm.models.glm5next.nvidia.specialized_decode.shared_expert",
 * SharedExpert.__call__, _GateUpKernel, _DownKernel and _group_scale:
 *   x-quant per 128 as in fme_moe_routed_fp8 (scale rule _group_scale);
 *   gate_up[t, n] = bf16(sum_b P[n, b] * (sx[b] * s13[n/128, b])), rows [0, I)
 *     are "gate", rows [I, 2I) are "up";
 *   h = bf16(silu(min(g, limit)) * clamp(u, -limit, limit)) (IEEE divide);
 *   h-quant per 128 by _group_scale (ue8m0 per flag), q = e4m3(h * (1 / sh));
 *   out[t, m] = bf16(sum_b P[m, b] * (sh[b] * s2[m/128, b])).
 *
 * Arguments: x [M, H] BF16; w13 [2I, H] E4M3; s13 [2I/128, H/128] FP32;
 *   w2 [H, I] E4M3; s2 [H/128, I/128] FP32 (fme_ue8m0_unpack converts packed
 *   UE8M0 scales); limits as fme_moe_routed_fp8 (E = 1, top_k = 1).
 *   gate_up: optional [M, 2I] BF16 output of the gate/up GEMV (NULL: not
 *   written). out [M, H] BF16.
 */
int fme_shared_expert_fp8(const void* x, const uint8_t* w13, const float* s13, const uint8_t* w2,
                          const float* s2, int M, int H, int I, float limit, int ue8m0,
                          void* gate_up, void* out, void* workspace, size_t workspace_bytes,
                          void* stream);

size_t fme_shared_expert_fp8_workspace(int M, int H, int I);

/*
 * Routed experts and shared expert of one FP8 decode layer in one launch.
 *
 * Sources: the routed part is fme_moe_routed_fp8 ("mega_moe"), the shared
 * part fme_shared_expert_fp8 ("shared_expert"), each with its own rounding
 * rules, weight layout (routed: up rows first; shared: gate rows first) and
 * clamp. The "shared_expert" page runs its two GEMVs as separate small kernels
 * beside the mega MoE kernel, sharing its SMs; here, up to 16 tokens, the
 * shared expert is one more unit of work in the routed kernel's schedule
 * (the first), so its 44 MB of weights stream in the same pass as the routed
 * experts' and no second launch or GEMM1 -> GEMM2 drain is paid for it. Above
 * 16 tokens its per-byte work (every token on one unit) would hold up the
 * launch, and the call issues two launches on the stream: the shared expert
 * alone, then the routed experts. Every token routes to it.
 *
 * Arguments: those of fme_moe_routed_fp8 (x, logits, bias, routed weights,
 * M, H, I, E, top_k, limit, scale, ue8m0, out, ids, weights), plus the shared
 * expert's shared_w13 [2I, H] E4M3, shared_s13 [2I/128, H/128] FP32,
 * shared_w2 [H, I] E4M3, shared_s2 [H/128, I/128] FP32, its clamp
 * shared_limit (> 0, +inf allowed) and scale flag shared_ue8m0, and its
 * output shared_out [M, H] BF16. The shared expert has the routed experts'
 * H and I. ids and weights equal those of fme_moe_routed_fp8 bit for bit;
 * out and shared_out meet the same tolerances. Up to 16 tokens they can differ
 * from the separate calls in the last bit of a few elements: the K blocks of a
 * tile are split over CTAs by the total work, which the extra unit changes,
 * and that changes the FP32 summation order.
 * workspace / workspace_bytes: see fme_moe_layer_fp8_workspace.
 */
int fme_moe_layer_fp8(const void* x, const void* logits, int logits_dtype, const float* bias,
                      const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                      int M, int H, int I, int E, int top_k, float limit, float scale, int ue8m0,
                      const uint8_t* shared_w13, const float* shared_s13, const uint8_t* shared_w2,
                      const float* shared_s2, float shared_limit, int shared_ue8m0, void* out,
                      int32_t* ids, float* weights, void* shared_out, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Workspace bytes fme_moe_layer_fp8 needs for these sizes (0 on bad sizes). */
size_t fme_moe_layer_fp8_workspace(int M, int H, int I, int E, int top_k);

/*
 * Local finalize: y[t] = bf16(sum over r = 0 .. top_k-1, in that order, of
 * weights[t, r] * out[t * top_k + r], plus shared_out[t] when given).
 *
 * Sources: "vllm.models.glm5next.nvidia.specialized_decode.mega_moe" (the
 * routed kernel returns unweighted rows t * top_k + r and the routing weights,
 * combined by a finalize step) and "vllm.models.kimi_k3.nvidia.
 * specialized_decode.cutedsl.moe.ep.comm" (EpCombine: the routing-weighted
 * sum, an FP32 sum in a fixed order, rounded once to BF16). Each product and
 * each sum is one FP32 rounding (no fused multiply-add); the shared row is
 * added after the routed sum; one BF16 rounding at the end.
 *
 * Arguments: out [M * top_k, H] BF16 (the routed call's out), weights
 * [M, top_k] FP32 (its weights), shared_out [M, H] BF16 or NULL (the shared
 * expert's out), y [M, H] BF16. 1 <= M <= 2^20, H a positive multiple of 8,
 * 1 <= top_k <= 32. out, shared_out and y 16-byte aligned, weights 4-byte
 * aligned; y must not overlap the inputs. Caller-owned buffers, no
 * workspace. Asynchronous on `stream`; the launch allows programmatic
 * dependent launch and waits for the preceding kernel before reading.
 * Returns FME_OK, FME_EINVAL, FME_EALIGN or FME_ECUDA.
 */
int fme_moe_finalize(const void* out, const float* weights, const void* shared_out, int M, int H, int top_k,
                     void* y, void* stream);

/*
 * MXFP8 quantisation of BF16 rows (the expert-parallel dispatch's quantiser,
 * single-GPU form).
 *
 * Source: "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.comm"
 * (EpDispatch: BF16 latent -> MXFP8, two threads per 32-value block, one E8M0
 * scale per 32 values in row order). The page does not print its exponent
 * rule; this follows the OCP MX rule: shared exponent floor(log2(amax)) - 8
 * (8 = the largest E4M3 exponent), clamped to [-127, 127], -127 for a zero
 * (or subnormal) amax; each value times 2^-exponent, E4M3 round-to-nearest-
 * even saturating at +-448; scale byte = exponent + 127.
 *
 * Arguments: x [T, H] BF16, q [T, H] E4M3 bytes, scales [T, H/32] bytes.
 * 1 <= T <= 2^20, H a positive multiple of 32. x and q 16-byte aligned.
 * Caller-owned buffers; asynchronous on `stream` (PDL launch).
 * Returns FME_OK, FME_EINVAL, FME_EALIGN or FME_ECUDA.
 */
int fme_mxfp8_quantize(const void* x, int T, int H, uint8_t* q, uint8_t* scales, void* stream);

/*
 * The combine's reduction and RMSNorm, single-GPU form.
 *
 * Source: "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.comm"
 * (EpCombine, rms_rstd): per token, the FP32 sum of the N partial rows in rank
 * order, rounded once to BF16 (the routed latent); then vLLM's RMSNorm of it:
 * FP32 sum of squares, rstd = rsqrt(sum / H + eps) (IEEE divide, approximate
 * reciprocal square root, as the page), out = bf16((x * rstd) * gamma).
 *
 * Arguments: partials [T, N, H] BF16 (row t * N + d = rank d's partial of
 * token t), gamma [H] BF16, eps >= 0 (the page: 1e-5), latent [T, H] BF16 and
 * normed [T, H] BF16 outputs. 1 <= N <= 1024, H a multiple of 8 up to 8192.
 * Every pointer 16-byte aligned; outputs must not overlap inputs.
 * Caller-owned buffers; asynchronous on `stream` (PDL launch).
 * Returns FME_OK, FME_EINVAL, FME_EALIGN or FME_ECUDA.
 */
int fme_combine_rmsnorm(const void* partials, int T, int N, int H, const void* gamma, float eps, void* latent,
                        void* normed, void* stream);

/*
 * Packed UE8M0 block scales -> FP32 block scales.
 *
 * Source: "vllm.models.glm5next.nvidia.specialized_decode.shared_expert",
 * block_scales: packed int32 [n, k/512], byte g % 4 of column g // 4 holds the
 * exponent of K group g; dst [n/128, k/128] FP32 with bits exponent << 23.
 * The exponent must be the same on all 128 rows of a row block: the kernel
 * reads row 128*i of each block and, when check != 0, compares every row and
 * sets *mismatch (device int, may be NULL when check == 0) to 1 on any
 * difference. n and k multiples of 128 and 512.
 */
int fme_ue8m0_unpack(const int32_t* packed, int n, int k, float* dst, int check, int* mismatch,
                     void* stream);

/*
 * NVFP4 slot MoE over the local experts [e0, e0 + L).
 *
 * Source: "nvfp4-megamoe-kernel README.md" (slot representation; Data Formats;
 * Bugs Found & Fixed 2, 4, 6, 7). A slot is a (token, pick) pair whose expert
 * is local; other picks are dropped. Per slot s of token t, local expert le:
 *   x-quant per 16: sc = e4m3(amax / 6) (stored UE4M3, also the divisor),
 *     q = e2m1(x / sc) (zeros when sc decodes to 0);
 *   g1[n] = bf16(sum_k dq(q_k) dq(W13[le, n, k])), dq = E2M1 value times its
 *     group-16 UE4M3 scale; rows [0, N) "gate", [N, 2N) "up";
 *   h = bf16(silu(min(gate, limit)) * clamp(up, -limit, limit)) per slot;
 *   h re-quantised like x; o[m] = bf16(sum_j dq(qh_j) dq(W2[le, m, j]));
 *   y[t, m] = bf16(sum over t's local slots, ascending pick, of
 *     topk_weights[t, r] * o[m]) accumulated in FP32: the routing weights
 *     are applied exactly once. Tokens with no local slot get zeros.
 * Arguments: x [M, H] BF16; topk_ids [M, top_k] int32 (global ids; negative
 *   or out-of-range ids are simply non-local); topk_weights [M, top_k] FP32;
 *   w13 [L, 2N, H/2] packed E2M1 (element 2i in the low nibble), s13
 *   [L, 2N, H/16] UE4M3 bytes; w2 [L, H, N/2], s2 [L, H, N/16]; limit > 0
 *   (+inf: no clamp). M in [1, 64], H and N multiples of 128 and <= 8192,
 *   L in [1, 1024], top_k in [1, 32]; a token's ids must be distinct.
 *   y [M, H] BF16.
 */
int fme_moe_routed_nvfp4(const void* x, const int32_t* topk_ids, const float* topk_weights,
                         const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                         const uint8_t* s2, int M, int H, int N, int L, int e0, int top_k,
                         float limit, void* y, void* workspace, size_t workspace_bytes,
                         void* stream);

size_t fme_moe_routed_nvfp4_workspace(int M, int H, int N, int L, int top_k);

/*
 * NVFP4 slot MoE with the routing fused in: fme_moe_routed_nvfp4 whose picks
 * come from router logits instead of the caller.
 *
 * Sources: the slot MoE as fme_moe_routed_nvfp4 ("nvfp4-megamoe-kernel
 * README.md"); the routing is the routed FP8 kernel's ("mega_moe"
 * _MegaKernel.top_k_pick): sigmoid scores, score + bias selects the top_k
 * experts (ties to the lower id) in descending order, weights = score / (FP32
 * sum of the picked scores in pick order) * scale. The page's NVFP4 pipeline
 * receives its picks from elsewhere; this entry computes them in the same
 * launch, every CTA for all tokens.
 *
 * Arguments: those of fme_moe_routed_nvfp4 without topk_ids / topk_weights,
 * plus logits [M, E] (logits_dtype FME_F32 or FME_BF16), bias [E] FP32, the
 * router's expert count E (1 .. 1024, with 0 <= e0 and e0 + L <= E), scale,
 * and the outputs ids [M, top_k] int32 and weights [M, top_k] FP32 (every
 * pick, local or not). top_k <= min(32, E). y, workspace, errors: as
 * fme_moe_routed_nvfp4 (same workspace size function; the two entries may
 * share a workspace).
 */
int fme_moe_layer_nvfp4(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
                        const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, int M, int H, int N, int L, int E,
                        int e0, int top_k, float scale, float limit, void* y, int32_t* ids, float* weights,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Zero a workspace (cudaMemsetAsync on stream). */
int fme_workspace_clear(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Read and clear the device error word of a workspace (synchronises stream).
 * *code receives 0 or a bit set: 1 = a ring wait timed out, 2 = a cross-CTA
 * wait timed out, 4 = the producer could not drain its copies, 8 = an output
 * row index fell outside its tensor (the write was skipped). Returns
 * FME_ETIMEOUT when *code != 0, FME_OK otherwise.
 */
int fme_workspace_error(void* workspace, int* code, void* stream);

/*
 * Self-test of the device-side bounded waits (no counterpart in the pages,
 * whose flag waits poll without a limit). Launches one small kernel that
 * waits, with the same primitives and a timeout_ms limit as the layer kernels,
 * on a flag nobody sets (workspace byte 256, which must be zero) and on an
 * mbarrier nobody arrives at. Both waits give up and set error bits 2 and 1
 * of the workspace error word; the GPU context stays usable. Read the result
 * with fme_workspace_error. workspace_bytes >= 512, timeout_ms in [1, 10000].
 */
int fme_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int timeout_ms, void* stream);

/* Number of streaming multiprocessors the kernels size their grids to. */
int fme_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FME_H_ */
