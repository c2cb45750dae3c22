/*
 * moe_gb300.h -- C ABI of a single-GPU (GB300, sm_103a) library that runs the forward pass of
 * a mixture-of-experts (MoE) layer whose expert weights are stored quantized.
 *
 * The pass: top-k routing with a renormalised softmax, permutation of (token, slot) rows by
 * expert, a grouped gate/up GEMM over packed weights, SiLU(gate) * up, a grouped down GEMM,
 * and the routing-weighted combine back to token order.
 *
 * Weight formats (model-card pages, cited by page title and section):
 *   MOE_FMT_FP8_B128_W8A16  clef-omni-fp8, "What was quantized" / "Recipe": E4M3 weights, one
 *                           fp32 scale per 128x128 tile (scale = 448/amax, stored inverted as
 *                           weight_scale_inv); bf16 activations.
 *   MOE_FMT_INT4_G128_W4A16 clef-omni-int4, "What was quantized": symmetric INT4, group 128
 *                           along K, auto_gptq packing; bf16 activations.
 *   MOE_FMT_NVFP4_W4A16     clef-omni-NVFP4, "How it was made": E2M1 codes two per byte, one
 *                           E4M3 scale per 16 weights, one fp32 global scale 448*6/amax per
 *                           expert matrix; bf16 activations.
 *   MOE_FMT_NVFP4_W4A4      the same weights with activations quantized to NVFP4 at run time
 *                           (clef-flash-NVFP4-Hybrid, layer table: 16-element groups, FP8 group
 *                           scales, one fp32 global scale), here one global scale per row.
 *   MOE_FMT_BF16            unquantized bf16 weights and activations through the same routing,
 *                           GEMM and combine kernels: the comparison point every quantized
 *                           checkpoint is measured against (clef-omni-fp8, "Which Clef-Omni quant
 *                           should I use?": the BF16 original is the reference row).
 *   MOE_FMT_FP8_B128_W8A8   the FP8 block weights of MOE_FMT_FP8_B128_W8A16 with activations
 *                           quantized to E4M3 at run time, one fp32 scale per 1x128 group of a
 *                           row (clef-omni-fp8, "What was quantized": serving engines may run the
 *                           FP8 experts this way); x and the gated intermediate h both.  Needs H
 *                           a multiple of 256 (MOE_ERR_UNSUPPORTED otherwise).
 *
 * Conventions for every call:
 *   - Pointers marked (dev) are device pointers; (host) are host pointers.  All memory is owned
 *     by the caller: the library never allocates, frees or synchronises inside the forward
 *     pass, and enqueues work only on the stream it is given.
 *   - Argument errors are reported synchronously by the return value and nothing is enqueued.
 *     MOE_ERR_CUDA means a CUDA launch or copy failed; cudaGetLastError() has the reason.
 *   - Device-side failures (a bounded wait that ran out, an index out of range) set an error
 *     word inside the workspace; moe_get_device_error() reads it.
 *   - Shapes: H and I are multiples of 128; 1 <= top_k <= min(E, 8); E <= 256; T >= 0.
 *   - bf16 tensors are passed as void* holding IEEE bfloat16 values.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = the legacy default stream */

typedef enum {
  MOE_FMT_FP8_B128_W8A16 = 1,
  MOE_FMT_INT4_G128_W4A16 = 2,
  MOE_FMT_NVFP4_W4A16 = 3,
  MOE_FMT_NVFP4_W4A4 = 4,
  MOE_FMT_BF16 = 5,
  MOE_FMT_FP8_B128_W8A8 = 6
} moe_format_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, bad format, k out of range */
  MOE_ERR_UNSUPPORTED = 2,  /* valid request this build cannot run (e.g. no sm_103a device) */
  MOE_ERR_WORKSPACE = 3,    /* workspace smaller than moe_workspace_size() asked for */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call failed */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device wait gave up (reported by moe_get_device_error) */
  MOE_ERR_DEVICE_FAULT = 6  /* a device-side bounds check fired (reported by moe_get_device_error) */
} moe_status_t;

/* Canonical tensors inside a packed-expert buffer (index into moe_packed_desc_t arrays).
 * Per format, for all E experts back to back ("gu" = fused gate/up [2I, H] with gate rows
 * 0..I-1 then up rows I..2I-1, "d" = down [H, I]; torch Linear orientation [out, in]):
 *   FP8 (W8A16 and W8A8):
 *          GU_A = codes u8 [E, 2I, H]      GU_B = scale_inv f32 [E, 2I/128, H/128]
 *          D_A  = codes u8 [E, H, I]       D_B  = scale_inv f32 [E, H/128, I/128]
 *   INT4:  GU_A = qweight i32 [E, H/8, 2I] GU_B = scales f16 [E, H/128, 2I]
 *          D_A  = qweight i32 [E, I/8, H]  D_B  = scales f16 [E, I/128, H]
 *          (nibble j of qweight word (kr, n) holds k = 8*kr + j; code = q + 8)
 *   NVFP4: GU_A = weight_packed u8 [E, 2I, H/2] (element 2i in the low nibble)
 *          GU_B = weight_scale E4M3 [E, 2I, H/16]
 *          D_A  = weight_packed u8 [E, H, I/2]  D_B = weight_scale E4M3 [E, H, I/16]
 *          GU_GS / D_GS = weight_global_scale f32 [E] (the quantize multiplier 2688/amax)
 *   BF16:  GU_A = bf16 [E, 2I, H]               D_A = bf16 [E, H, I]  (the weights as given)
 *   NVFP4 W4A4 also carries both matrices as a tensor-core operand image: the same codes and
 *   scales rearranged into the exact shared-memory image that one block-scaled MMA step reads,
 *   so that each (pair of 128-row tiles, 256-column chunk) arrives in one bulk copy:
 *          GU_IMG = u8 [E, I/128, C(H), 36864]   D_IMG = u8 [E, ceil(H/256), C(I), 36864]
 *   (C(K) = ceil(K/256) chunks).  Block [e, p, c]: tile 0 = rows r0 .. r0+127, tile 1 = rows
 *   r1 .. r1+127 (gate/up: r0 = 128p gate rows, r1 = I + 128p the matching up rows; down:
 *   r0 = 256p, r1 = 256p + 128, a tile past H all zero); bytes [16384 g, 16384 g + 16384) hold
 *   tile g's codes of columns 256c .. 256c+255, row l's 128 bytes at 128 l with 16-byte piece j
 *   stored at piece j ^ (l % 8) (the 128-byte swizzle); bytes [32768 + 2048 g, + 2048) hold
 *   tile g's scales in the order tensor memory takes them: byte 512 s + 16 l + 4 j + i = the
 *   scale of row 32 j + l, 16-block 16c + 4s + i.  Columns past K (a last half chunk) are zero.
 *   Written by moe_pack_experts next to the canonical tensors; not part of the checkpoint format.
 *   NVFP4 W4A16 carries its codes and scales again as the bf16 converter's weight image:
 *          GU_IMG = u8 [E, H/128, 2I/128, 9216]   D_IMG = u8 [E, I/128, H/128, 9216]
 *   Block [e, c, b] = one 128-row tile (gate/up: gate rows 64b .. 64b+63, then up rows
 *   I+64b .. I+64b+63; down: rows 128b .. 128b+127) of columns 128c .. 128c+127: row l's 64 code
 *   bytes at 64 l with 16-byte piece p stored at piece p ^ ((l / 2) % 4), then at 8192 + 8 l the
 *   row's 8 E4M3 scales.  Each little-endian 32-bit code word (eight codes; element k = nibble k
 *   of the canonical word, code bits m, e0, e1, s) is re-ordered so that bits (m, e0, e1, s) of
 *   element k sit at bits
 *   k=0: 0,1,2,9  k=1: 16,17,18,25  k=2: 4,5,6,13  k=3: 20,21,22,29
 *   k=4: 10,11,12,19  k=5: 26,27,28,3  k=6: 14,7,8,15  k=7: 30,23,24,31.
 *   Also written by moe_pack_experts.
 * Every tensor starts on a 256-byte boundary of the packed buffer. */
enum {
  MOE_T_GU_A = 0,
  MOE_T_GU_B = 1,
  MOE_T_D_A = 2,
  MOE_T_D_B = 3,
  MOE_T_GU_GS = 4,
  MOE_T_D_GS = 5,
  MOE_T_GU_IMG = 6,
  MOE_T_D_IMG = 7,
  MOE_T_COUNT = 8
};

typedef struct {
  int32_t fmt;                   /* moe_format_t */
  int32_t E, H, I;               /* experts, hidden size, expert intermediate size */
  uint64_t bytes;                /* total size of the packed buffer */
  uint64_t offset[MOE_T_COUNT];  /* byte offset of each canonical tensor (0 if absent) */
  uint64_t size[MOE_T_COUNT];    /* byte size of each canonical tensor (0 if absent) */
} moe_packed_desc_t;

/* Fill *desc with the packed layout for (fmt, E, H, I).  Host only; no CUDA calls.
 * The tensors and their sizes are the checkpoint tensors the pages name for each format:
 * weight + weight_scale_inv (clef-omni-fp8, "What was quantized"), qweight + scales in
 * auto_gptq packing (clef-omni-int4, "What was quantized"), weight_packed + weight_scale +
 * weight_global_scale (clef-omni-NVFP4, "How it was made"), for the fused gate/up and the down
 * matrix of each expert (clef-omni-int4, "How this checkpoint runs": the experts of a layer are
 * stacked and run as one grouped matmul).
 * Errors: MOE_ERR_INVALID_ARG for a null desc, an unknown format, E outside 1..256, or H, I not
 * positive multiples of 128 (desc is then zeroed apart from the echoed arguments). */
moe_status_t moe_packed_size(int fmt, int E, int H, int I, moe_packed_desc_t* desc);

/* Quantize and pack bf16 expert weights on the GPU (stream-ordered, asynchronous).
 *   w_gate_up (dev) bf16 [E, 2I, H]; w_down (dev) bf16 [E, H, I]; packed (dev) desc->bytes,
 *   256-byte aligned; all three caller-owned and not modified apart from packed.
 * Results are bit-identical to the quantizers the pages give (per-tile / per-group / per-block
 * amax scaling, round-to-nearest-even): FP8 per 128x128 tile, s = 448/amax (clef-omni-fp8,
 * "Recipe"); INT4 per 128-group along K, fp16 scale amax/7, codes + 8 (clef-omni-int4, "What was
 * quantized"); NVFP4 16-element blocks, E4M3 block scales, one fp32 global scale per matrix with
 * gate and up sharing it (clef-omni-NVFP4, "How it was made").
 * Errors: MOE_ERR_INVALID_ARG for a bad desc (or one not produced by moe_packed_size for its
 * own arguments), a null or misaligned pointer; MOE_ERR_UNSUPPORTED on a device other than
 * sm_103; MOE_ERR_CUDA if a launch fails.  Nothing is enqueued on an argument error. */
moe_status_t moe_pack_experts(const moe_packed_desc_t* desc, const void* w_gate_up, const void* w_down,
                              void* packed, moe_stream_t stream);

/* Bytes of device workspace moe_layer_forward needs for T tokens and top_k (host only).
 * The same size also serves moe_debug_route and moe_get_device_error.  It holds the routing
 * tables, the permutation and the intermediate h of the grouped matmuls (clef-omni-int4, "How
 * this checkpoint runs": route, group the tokens by expert, one grouped matmul per projection).
 * Errors: MOE_ERR_INVALID_ARG for a bad desc, a null bytes, T < 0 or top_k outside 1..min(E, 8). */
moe_status_t moe_workspace_size(const moe_packed_desc_t* desc, int T, int top_k, size_t* bytes);

/* The forward pass of one MoE layer (clef-omni-int4, "How this checkpoint runs": the routed
 * experts of a layer run as one grouped matmul; clef-omni-fp8, "How this checkpoint runs": the
 * same for the FP8 experts; the gated-MLP experts of the Qwen3-MoE backbone, clef-omni-NVFP4,
 * "Credits"), on `stream` (asynchronous; no host synchronisation, no allocation):
 *   x (dev) bf16 [T, H]; router_logits (dev) f32 [T, E]; packed (dev) from moe_pack_experts;
 *   out (dev) bf16 [T, H], must not alias x; workspace (dev) >= moe_workspace_size bytes,
 *   256-byte aligned, contents need not be initialised and are overwritten.
 * out[t] = sum_j w_tj * Wd_e (silu(Wg_e a_t) * (Wu_e a_t)), e = j-th routed expert of t,
 * w = softmax over the top-k logits, a_t = x_t (W*A16) or its NVFP4 quantization (W4A4). */
moe_status_t moe_layer_forward(const void* x, const float* router_logits, int T, const moe_packed_desc_t* desc,
                               const void* packed, int top_k, void* out, void* workspace, size_t ws_bytes,
                               moe_stream_t stream);

/* NVFP4 W4A4 with static activation scales (clef-flash-NVFP4-Hybrid, "Quantization details":
 * one FP32 global scale per tensor, the activation scales calibrated ahead of time): the same
 * pass as moe_layer_forward, but every row of x is quantized with the one global scale
 * act_gs[0] and every row of h with act_gs[1] (the quantize multiplier, as for the weights:
 * codes = E2M1(value / (E4M3 block scale / gs))); blocks beyond the calibrated range saturate.
 * h is quantized inside the gate/up GEMM and never written in bf16.
 *   act_gs (dev) f32 [2], 4-byte aligned, read by the kernels of this call (stream-ordered).
 * MOE_ERR_INVALID_ARG for any other format or a null act_gs; otherwise as moe_layer_forward. */
moe_status_t moe_layer_forward_static_act(const void* x, const float* router_logits, int T,
                                          const moe_packed_desc_t* desc, const void* packed, int top_k,
                                          const float* act_gs, void* out, void* workspace, size_t ws_bytes,
                                          moe_stream_t stream);

/* Calibration of those static scales on one batch (W4A4, T >= 1):
 * act_gs[0] = 2688 / max |x| over the batch; then x is quantized with it, the gate/up GEMM runs,
 * and act_gs[1] = 2688 / max |h| over every routed row (h in bf16); each amax is clamped to
 * >= 1e-12 as in the dynamic rule.  No output is written; the workspace is that of
 * moe_layer_forward.  act_gs (dev) f32 [2], 4-byte aligned, written stream-ordered.
 * MOE_ERR_INVALID_ARG for T < 1, a null act_gs or a format other than MOE_FMT_NVFP4_W4A4. */
moe_status_t moe_calibrate_act_scales(const void* x, const float* router_logits, int T, const moe_packed_desc_t* desc,
                                      const void* packed, int top_k, float* act_gs, void* workspace,
                                      size_t ws_bytes, moe_stream_t stream);

/* Bytes of workspace moe_layer_forward_host needs: moe_workspace_size plus device staging for
 * x, the logits and out (host only).  Same errors as moe_workspace_size. */
moe_status_t moe_workspace_size_host_io(const moe_packed_desc_t* desc, int T, int top_k, size_t* bytes);

/* moe_layer_forward (same passage) with HOST activations: copies x_host bf16 [T, H] and
 * logits_host f32 [T, E] into the workspace, runs the layer, copies the result to out_host
 * bf16 [T, H], all on `stream` and asynchronously (use pinned host memory for overlap; the
 * caller synchronises before reading out_host).  packed stays on the device.  The workspace
 * must have moe_workspace_size_host_io bytes.  Errors as moe_layer_forward. */
moe_status_t moe_layer_forward_host(const void* x_host, const float* logits_host, int T,
                                    const moe_packed_desc_t* desc, const void* packed, int top_k,
                                    void* out_host, void* workspace, size_t ws_bytes, moe_stream_t stream);

/* Synchronise `stream`, then read and clear the device error word kept in `workspace`.
 * *code receives MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_FAULT.  The pages have no
 * counterpart: it reports this library's own bounded device waits and bounds checks.
 * Errors: MOE_ERR_INVALID_ARG for a null pointer; MOE_ERR_CUDA if the copy or sync fails. */
moe_status_t moe_get_device_error(void* workspace, moe_stream_t stream, int32_t* code);

/* A static English description of a status code (library bookkeeping, no page counterpart). */
const char* moe_status_string(int status);

/* ---- inspection views of individual steps (same kernels as the forward pass) ---------- */

/* Routing and permutation alone, the first step of moe_layer_forward: the router's logits are
 * left unquantized (clef-omni-fp8, page header and "What was quantized"), and grouping rows by
 * expert feeds the grouped matmul (clef-omni-int4, "How this checkpoint runs").  Outputs:
 * topk_idx i32 [T, k] (descending logits, ties to the lower expert), topk_w f32 [T, k]
 * (renormalised softmax over the k selected logits), offsets i32 [E+1], perm i32 [T*k]
 * (row r holds t*k + j, rows sorted by expert, token, slot), inv i32 [T*k] (row of t*k + j).
 * All (dev), caller-owned.  workspace as for moe_layer_forward (256-byte aligned).
 * Errors: MOE_ERR_INVALID_ARG for bad sizes or null pointers; MOE_ERR_WORKSPACE if ws_bytes is
 * too small; MOE_ERR_UNSUPPORTED off sm_103; MOE_ERR_CUDA if a launch or copy fails. */
moe_status_t moe_debug_route(const float* router_logits, int T, int E, int top_k, int32_t* topk_idx,
                             float* topk_w, int32_t* offsets, int32_t* perm, int32_t* inv, void* workspace,
                             size_t ws_bytes, moe_stream_t stream);

/* Dequantize one packed matrix to f32 (dev) [N, K]: which = 0 fused gate/up, 1 down: the
 * pages' dequantize-then-matmul step (clef-omni-fp8, "How this checkpoint runs"; clef-omni-NVFP4,
 * "How it was made"), here only an inspection view since the GEMMs dequantize in place.
 * Values are bit-identical to the format's dequantization rule:
 *   FP8 code * scale_inv; INT4 (code - 8) * scale; NVFP4 (e2m1 * e4m3) / global_scale.
 * Errors: MOE_ERR_INVALID_ARG for a bad desc, expert or which, or a null pointer. */
moe_status_t moe_debug_dequant(const moe_packed_desc_t* desc, const void* packed, int expert, int which,
                               float* out, moe_stream_t stream);

/* Dynamic NVFP4 quantization of bf16 rows x (dev) [T, H]: codes u8 [T, H/2], scales E4M3
 * [T, H/16], gs f32 [T] = 2688 / max(amax(row), 1e-12).  Bit-identical to the W4A4 rule (the
 * weight recipe of clef-omni-NVFP4, "How it was made", applied per activation row; NVFP4
 * activations: clef-flash-NVFP4-Hybrid, "Quantization details").  x 16-byte aligned.
 * Errors: MOE_ERR_INVALID_ARG for H not a multiple of 16 or a null pointer. */
moe_status_t moe_debug_quant_act(const void* x, int T, int H, uint8_t* codes, uint8_t* scales, float* gs,
                                 moe_stream_t stream);

/* The same with one static global scale for every row: gs_static (dev) f32 [1] (the quantize
 * multiplier; the calibrated per-tensor activation scale of clef-flash-NVFP4-Hybrid,
 * "Quantization details"); codes and scales as above (what moe_layer_forward_static_act feeds
 * the GEMMs).  Errors as moe_debug_quant_act. */
moe_status_t moe_debug_quant_act_static(const void* x, int T, int H, const float* gs_static, uint8_t* codes,
                                        uint8_t* scales, moe_stream_t stream);

/* Dynamic FP8 quantization of bf16 rows x (dev) [T, H] as MOE_FMT_FP8_B128_W8A8 applies it
 * (clef-omni-fp8, "What was quantized" and "Recipe", the tile rule on a 1x128 group): per group
 * of 128 consecutive elements of a row, s = 448 / max(amax, 1e-12), codes E4M3(v * s) u8 [T, H]
 * (round to nearest even, saturating at 448), scale_inv f32 [T, H/128] = 1 / s.  H a multiple
 * of 128, x 16-byte aligned, codes and scale_inv 4-byte aligned, all caller-owned; otherwise
 * MOE_ERR_INVALID_ARG and nothing is enqueued.  Asynchronous on stream. */
moe_status_t moe_debug_quant_act_fp8(const void* x, int T, int H, uint8_t* codes, float* scale_inv,
                                     moe_stream_t stream);

/* Test-only check of device failure detection (no page counterpart): enqueues one thread that
 * waits on a barrier nothing completes, through the bounded wait every GEMM kernel uses (about 2*10^9 SM cycles,
 * roughly one second).  When the wait gives up it records MOE_ERR_DEVICE_TIMEOUT in the error
 * word of workspace (dev, 256-byte aligned, any workspace this library sized) and returns;
 * moe_get_device_error() then reports it, and the CUDA context stays usable.  Returns
 * MOE_ERR_INVALID_ARG for a null or misaligned workspace. */
moe_status_t moe_debug_wait_timeout(void* workspace, moe_stream_t stream);

/* ---- routing without any caller workspace ----------------------------------------------- */

/* The pages have no counterpart to this entry point; it exists for callers that cannot obtain
 * device memory at this point: a plugin or callback run by a host engine that owns every device
 * allocation and gives it no scratch, or a serving loop with a memory pool fixed at start-up
 * where a cudaMalloc (and the device-wide synchronisation it brings) would stall other streams.
 *
 * Same results as moe_debug_route (same kernels), but the routing scratch lives in a static
 * device array inside the library (MOE_ROUTE_NOALLOC_SCRATCH_BYTES, held on every GPU that
 * loads the library until the process exits).  The call allocates nothing and frees nothing.
 *   router_logits (dev) f32 [T, E]; topk_idx (dev) i32 [T, k]; topk_w (dev) f32 [T, k];
 *   offsets (dev) i32 [E+1]; perm (dev) i32 [T*k]; inv (dev) i32 [T*k]; all caller-owned.
 * Limits: T <= MOE_ROUTE_NOALLOC_MAX_TOKENS, E <= 256, top_k <= 8.  Larger T returns
 * MOE_ERR_WORKSPACE ("workspace too small") before anything is enqueued.
 * The first call on each device resolves the array's device address (cudaGetSymbolAddress with
 * that device current) and caches it: make that first call before any stream capture begins.
 * All calls share the one array, which keeps the last call's contents (each call writes all it
 * reads); calls whose work overlaps on the GPU, e.g. on two streams, race on it. */
#define MOE_ROUTE_NOALLOC_MAX_TOKENS 2048
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES (512u * 1024u)
moe_status_t moe_route_noalloc(const float* router_logits, int T, int E, int top_k, int32_t* topk_idx,
                               float* topk_w, int32_t* offsets, int32_t* perm, int32_t* inv, moe_stream_t stream);

/* ---- measurement hooks ------------------------------------------------------------------ */

/* Total number of CUDA kernels this library has enqueued in the calling process (all threads,
 * all devices) since it was loaded.  Memsets and copies are not counted.  Measurement only; no
 * page counterpart. */
uint64_t moe_kernel_launch_count(void);

/* Measurement only (no page counterpart).
 * Ask the next moe_layer_forward / moe_layer_forward_host call made by this host thread to
 * record `start` right before and `stop` right after the launches of one step, on the call's
 * stream (step 0 = grouped gate/up GEMM, 1 = grouped down GEMM).  The request is consumed by
 * that one call.  Events are cudaEvent_t passed as void*; pass NULL to cancel. */
moe_status_t moe_time_next_step(int step, void* start, void* stop);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
