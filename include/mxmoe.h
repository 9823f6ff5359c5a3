/*
 * mxmoe.h -- C ABI of a GB300 (sm_103a) W4A4 MXFP4 mixture-of-experts expert layer.
 *
 * The layer: bf16 tokens are quantised to packed E2M1 with one UE8M0 scale per 32
 * elements, bucketed by their top-k experts, multiplied with each expert's gate/up
 * weight (MXFP4) through a SwiGLU, requantised to MXFP4, multiplied with the
 * expert's down weight (MXFP4), and summed over the k experts with the routing
 * weights into a bf16 output.  Sources:
 *   - "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE (W4A4)": the
 *     packed FP4 x FP4 mega-MoE kernel on a DeepSeek-V4-Flash layer (hidden 4096,
 *     inter 2048, 256 experts, top-6), Appendix B.
 *   - prhub digest of SGLang PR #37279 ("升级 sgl-deep-gemm 至 0.1.7，MegaMoE 改用
 *     mma_type API 支持 MXFP4"): sections 实现拆解 items 1-4 and the mega_moe.py
 *     excerpt -- the explicit mma_type "mxf4xmxf4", the per-mma-type buffer,
 *     pre_dispatch(hidden, topk ids, topk weights, ..., num_tokens, group_size=32),
 *     the weight transform and the gran=16 gate/up interleave.
 *   - SGLang PR #48424, "DeepGEMM producers write FlashInfer's 128x4 scale layout":
 *     scales as 4-D int32 [ceil(rows/128), K/128, 32, 4]; live rows are a prefix.
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are CUDA device pointers, *_host host pointers.  Device
 *     buffers are allocated and freed by the caller; no hot entry point allocates.
 *   - Device pointers passed to kernels must be 16-byte aligned (256-byte for the
 *     prepared weights and the workspace); otherwise MOE_ERR_INVALID_ARG.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *     asynchronously and stream-ordered; only moe_check, moe_run_host and the
 *     moe_read_* debug calls synchronise.
 *   - A failing call returns a nonzero moe_status and records a message readable
 *     with moe_last_error() (per thread).  Nothing is enqueued after a failed
 *     argument check.
 *   - Element formats: E2M1 codes are packed two per byte, element 2i in the low
 *     nibble of byte i.  A scale byte b means 2^(b-127) (UE8M0).  The scale of a
 *     group of 32 is 2^e with e the smallest integer such that amax <= 6 * 2^e,
 *     clamped to [-127, 127]; elements round to the nearest E2M1 value, ties to
 *     the even code, and keep their sign.
 */
#ifndef MXMOE_H
#define MXMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MXMOE_API __attribute__((visibility("default")))
#else
#define MXMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
typedef int32_t moe_status;
enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* null/misaligned pointer, bad size or shape   */
    MOE_ERR_UNSUPPORTED = 2,         /* mma_type or mode that is not built           */
    MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < moe_workspace_size(dims)          */
    MOE_ERR_WORKSPACE_MISMATCH = 4,  /* workspace initialised for other dims/mma    */
    MOE_ERR_CUDA = 5,                /* a CUDA runtime/driver call failed            */
    MOE_ERR_ROUTING = 6,             /* device saw topk ids outside [0, E)           */
    MOE_ERR_TIMEOUT = 7              /* a device wait ran past its limit             */
};

/* Operand types of the expert GEMMs (digest of PR #37279, items 1-4: the explicit
 * mma_type):
 *   MOE_MMA_MXF4xMXF4  "mxf4xmxf4": activations MXFP4 (packed E2M1, UE8M0 per 32),
 *                      W1 gate/up rows interleaved with gran=16 (even/odd).
 *   MOE_MMA_FP8xFP4    "fp8xfp4" (W4A8): activations MXFP8 (one E4M3 byte per
 *                      element, UE8M0 per 32; the scale 2^e with e the smallest
 *                      integer such that amax <= 448 * 2^e), W1 gate/up rows
 *                      interleaved with gran=8 ([gate 0..7, up 0..7, gate 8..15, ..]).
 *   MOE_MMA_NVF4xNVF4  NVFP4 throughout: packed E2M1 activations and weights with one
 *                      unsigned E4M3 scale per 16 elements (the E4M3 value nearest
 *                      to amax/6; elements fp32(x / scale) rounded to E2M1, ties to
 *                      even, saturating at 6; no per-tensor scale), gran=16.
 * The weights are MXFP4 in the first two (NVFP4 in the third: see
 * moe_quantize_nvfp4).  Every other value returns MOE_ERR_UNSUPPORTED. */
enum { MOE_MMA_MXF4xMXF4 = 1, MOE_MMA_FP8xFP4 = 2, MOE_MMA_NVF4xNVF4 = 3 };

/* Layer dimensions.  hidden H and inter I must be multiples of 128 (H >= 256);
 * 1 <= topk <= min(num_experts, 32); 1 <= num_experts <= 1024;
 * 1 <= max_tokens <= 65536 (the capacity a workspace is sized for). */
typedef struct moe_dims {
    int32_t hidden;
    int32_t inter;
    int32_t num_experts;
    int32_t topk;
    int32_t max_tokens;
    int32_t mma_type;
} moe_dims;

/* Message of the last failure on this thread ("" if none). */
MXMOE_API const char *moe_last_error(void);

/* Static name of a status code. */
MXMOE_API const char *moe_status_string(moe_status s);

/* Checks dims as described above.  Host only; no CUDA call. */
MXMOE_API moe_status moe_validate_dims(const moe_dims *dims);

/* Bytes of the prepared-weight blob moe_prepare_weights writes; 0 for bad dims.
 * Equal to the canonical bytes of both weights (each of the four sections rounded
 * up to 1 KiB) when K (hidden for W1, inter for W2) is a whole number of k-blocks
 * (256 elements; 128 for MOE_MMA_FP8xFP4); otherwise each code row is padded to
 * whole k-blocks.  Host only. */
MXMOE_API size_t moe_prepared_weights_size(const moe_dims *dims);

/* Bytes of the workspace for dims->max_tokens tokens; 0 for bad dims.  Host only.
 * (The pages' symmetric buffer sized by num_max_tokens_per_rank, one per
 * mma_type; this library runs on one GPU, so it is plain device memory.) */
MXMOE_API size_t moe_workspace_size(const moe_dims *dims);

/* Initialises a workspace: clears it and records dims and mma_type in its header
 * and in a host-side registry, so that later calls with other dims return
 * MOE_ERR_WORKSPACE_MISMATCH (the pages key their buffer cache on the dims and
 * mma_type for the same reason).  Must precede the first pre_dispatch on it. */
MXMOE_API moe_status moe_workspace_init(const moe_dims *dims, void *ws_dev, size_t ws_bytes,
                                        void *stream);

/* How pre_dispatch hands the quantised tokens to the layer (SGLang PR #48424,
 * Summary: "SIMT dispatch pull for FP4 activations"):
 *   MOE_DISPATCH_BUCKETED (default after moe_workspace_init): each token's row is
 *     copied to the row of every one of its assignments, expert-contiguous, and the
 *     layer loads token tiles from there with TMA.
 *   MOE_DISPATCH_PULL: each token's row is written once, and the layer gathers its
 *     experts' token tiles from those rows with asynchronous per-thread copies.
 * Both give the same results.  Set on an initialised workspace, before the
 * pre_dispatch whose forward should use it; MOE_ERR_INVALID_ARG for an unknown mode,
 * MOE_ERR_WORKSPACE_MISMATCH for a workspace moe_workspace_init has not seen,
 * MOE_ERR_UNSUPPORTED for MOE_DISPATCH_PULL on an fp8xfp4 or nvf4xnvf4 workspace
 * (pull is built for MXFP4 activations only). */
enum { MOE_DISPATCH_BUCKETED = 0, MOE_DISPATCH_PULL = 1 };
MXMOE_API moe_status moe_workspace_set_dispatch(void *ws_dev, int32_t mode);

/* Token tiles of the grouped GEMMs:
 *   MOE_TILES_WIDE:   up to 128 token rows a tile, expert segments padded to 128 rows.
 *   MOE_TILES_NARROW: up to 32 rows a tile (segments padded to 32); the layer then
 *                     keeps four stages of operands in flight instead of three,
 *                     which pays when experts hold few tokens (decode-sized loads).
 *   MOE_TILES_MEDIUM: up to 64 rows a tile (segments padded to 64), four stages where
 *                     shared memory allows (three for nvf4xnvf4).
 *   MOE_TILES_PAIR:   up to 192 rows a tile, each tile starting a 256-row span of the
 *                     expert's segment (the last one padded to 128 rows), each item of
 *                     the layer run by two SMs together (a 2-CTA cluster issuing M=256
 *                     tcgen05 MMAs over both SMs' shared memory: 1.6 times the FLOPs
 *                     per staged operand byte).  mxf4xmxf4 with the bucketed dispatch
 *                     and H a multiple of 256 only; otherwise it falls back to wide
 *                     tiles.  Slower than wide tiles on GB300 (one MMA-issuing thread
 *                     per two SMs), so MOE_TILES_AUTO never picks it.
 *   MOE_TILES_AUTO (default after moe_workspace_init): narrow when num_tokens * k <=
 *                     16 * num_experts, medium when <= 64 * num_experts, else wide.
 * The choice is made at each moe_pre_dispatch and holds for the forward that
 * follows; results are the same either way up to fp32 summation order.  The pull
 * dispatch always uses wide tiles.  MOE_ERR_INVALID_ARG for an unknown mode,
 * MOE_ERR_WORKSPACE_MISMATCH for a workspace moe_workspace_init has not seen. */
enum { MOE_TILES_AUTO = 0, MOE_TILES_WIDE = 1, MOE_TILES_NARROW = 2, MOE_TILES_MEDIUM = 3,
       MOE_TILES_PAIR = 4 };
MXMOE_API moe_status moe_workspace_set_tiles(void *ws_dev, int32_t mode);

/* Quantises row-major fp32 src_dev [rows, K] (K % 32 == 0) to MXFP4 with the rule
 * above: codes_dev [rows, K/2], scales_dev [rows, K/32], both row-major.  A helper
 * for producing canonical MXFP4 weights on the device. */
MXMOE_API moe_status moe_quantize_mxfp4(const float *src_dev, int64_t rows, int32_t K,
                                        uint8_t *codes_dev, uint8_t *scales_dev, void *stream);

/* As moe_quantize_mxfp4 for NVFP4 (K % 16 == 0): codes_dev [rows, K/2], scales_dev
 * [rows, K/16] one E4M3 byte per 16 elements, with the rule of MOE_MMA_NVF4xNVF4.
 * Canonical NVFP4 weights for moe_prepare_weights under that mma_type. */
MXMOE_API moe_status moe_quantize_nvfp4(const float *src_dev, int64_t rows, int32_t K,
                                        uint8_t *codes_dev, uint8_t *scales_dev, void *stream);

/* Weight transform (the pages' transform_weights_for_mega_moe with mma_type
 * mxf4xmxf4).  Inputs are canonical MXFP4, row-major:
 *   w1_codes_dev [E, 2I, H/2], w1_scales_dev [E, 2I, H/32]   gate rows 0..I-1, up rows I..2I-1
 *   w2_codes_dev [E, H, I/2],  w2_scales_dev [E, H, I/32]
 *   (NVFP4 for nvf4xnvf4: scales [E, 2I, H/16] and [E, H, I/16], E4M3 bytes)
 * Output `prepared_dev` (prepared_bytes >= moe_prepared_weights_size): W1 rows
 * interleaved with gran=16 (each chunk of 16 gate and 16 up rows becomes
 * [gate even, up even, gate odd, up odd]; for fp8xfp4 gran=8: [gate 8, up 8]),
 * codes and scales alike.  Sections, each 1 KiB-aligned: W1 codes, W1 scales, W2
 * codes, W2 scales.  Codes are stored in k-block tiles, so that one weight slab's
 * k-block is one contiguous run: with kb = 128 bytes (64 for fp8xfp4) and
 * nkb = ceil(K / (2 kb)), byte j of row R (rows over all experts) sits at
 * ((R / 128 * nkb + j / kb) * 128 + R % 128) * kb + j % kb, and the bytes past a
 * row's end in a short last k-block are zero.  Scales are in the 128x4 block
 * layout.  Inputs are not modified; the caller may free them afterwards. */
MXMOE_API moe_status moe_prepare_weights(const moe_dims *dims, const uint8_t *w1_codes_dev,
                                         const uint8_t *w1_scales_dev, const uint8_t *w2_codes_dev,
                                         const uint8_t *w2_scales_dev, void *prepared_dev,
                                         size_t prepared_bytes, void *stream);

/* Quantise-and-bucket (the pages' mega_moe_pre_dispatch, group_size 32): MXFP4 or,
 * for fp8xfp4, MXFP8 token rows (see MOE_MMA_*).
 *   x_dev            bf16 [num_tokens, H] row-major, finite values
 *   topk_ids_dev     int32 [num_tokens, k]; ids outside [0, E) are skipped and
 *                    raise MOE_ERR_ROUTING at the next moe_check
 *   topk_weights_dev fp32 [num_tokens, k], used as given (no renormalisation)
 * num_tokens <= dims->max_tokens; num_tokens == 0 is a no-op.  Writes the
 * quantised token rows, per-expert counts and slots into the workspace.
 * Within an expert, slots are ordered by ascending token, then ascending k index. */
MXMOE_API moe_status moe_pre_dispatch(const moe_dims *dims, const void *x_dev,
                                      const int32_t *topk_ids_dev, const float *topk_weights_dev,
                                      int32_t num_tokens, void *ws_dev, size_t ws_bytes,
                                      void *stream);

/* The expert layer on the buffers of the last moe_pre_dispatch on this workspace
 * (same num_tokens): grouped gate/up GEMM with SwiGLU and requantisation to the
 * activation format of dims->mma_type,
 * grouped down GEMM, top-k weighted combine.  out_dev: bf16 [num_tokens, H].
 * Defined by: the digest of PR #37279, section 实现拆解 item 3 (_run_mega_routed, the
 * routed forward: pre_dispatch into the per-mma_type buffer, then the fused mega-MoE
 * kernel with activation "swiglu"), and "[deepseek-v4] Bump sgl-deep-gemm for packed
 * FP4xFP4 mega-MoE (W4A4)", Appendix B (that fused kernel: both expert GEMMs and the
 * combine in one launch, streaming every touched expert's packed FP4 weights).
 *   dims        the dims the workspace was initialised with (else
 *               MOE_ERR_WORKSPACE_MISMATCH)
 *   prepared_dev  the blob moe_prepare_weights wrote for these dims, 256-byte aligned
 *   ws_dev, ws_bytes  the workspace and its size in bytes (checked against
 *               moe_workspace_size; too small: MOE_ERR_WORKSPACE_TOO_SMALL)
 *   num_tokens  as passed to the last moe_pre_dispatch; 0 is a no-op
 * The workspace's fp32 accumulator and intermediate rows are overwritten; the
 * prepared weights are only read.
 * Calling it again without a new moe_pre_dispatch recomputes the same layer (the
 * library then clears the accumulator rows first). */
MXMOE_API moe_status moe_forward(const moe_dims *dims, const void *prepared_dev, void *ws_dev,
                                 size_t ws_bytes, void *out_dev, int32_t num_tokens, void *stream);

/* End-to-end call on HOST buffers: x_host (bf16 [T, H]), topk_ids_host and
 * topk_weights_host in, the bf16 result in out_host [T, H]; runs moe_pre_dispatch
 * and moe_forward and synchronises the stream.  Each page-locked buffer
 * (cudaHostAlloc, cudaHostRegister; 16-byte aligned) is read or written by the
 * kernels directly over the host link; any other buffer goes through a staging
 * area of the workspace with a copy. */
MXMOE_API moe_status moe_run_host(const moe_dims *dims, const void *prepared_dev, void *ws_dev,
                                  size_t ws_bytes, const void *x_host,
                                  const int32_t *topk_ids_host, const float *topk_weights_host,
                                  void *out_host, int32_t num_tokens, void *stream);

/* Synchronises `stream`, then reads and clears the workspace's device error
 * flags: MOE_ERR_ROUTING, MOE_ERR_TIMEOUT, or MOE_OK. */
MXMOE_API moe_status moe_check(void *ws_dev, void *stream);

/* ---- debug readback (tests only; synchronous, allocate nothing on the device) ----
 * Canonical views of what the last pre_dispatch/forward wrote for num_tokens
 * tokens.  Assignment a = t*k + j.  A null output pointer skips that output.
 *   counts_host        int32 [E]          tokens routed to each expert
 *   assign_slot_host   int32 [T*k]        workspace row of assignment a (-1: skipped)
 *   x_codes_host       uint8 [T*k, H/2]   quantised token row as stored for assignment a
 *                                         ([T*k, H]: one E4M3 byte each, for fp8xfp4)
 *   x_scales_host      uint8 [T*k, H/32]   ([T*k, H/16] E4M3 bytes for nvf4xnvf4)
 *   slot_token_host    int32 [T*k]        token recorded in row assign_slot[a] (check) */
MXMOE_API moe_status moe_read_dispatch(const moe_dims *dims, const void *ws_dev,
                                       int32_t num_tokens, int32_t *counts_host,
                                       int32_t *assign_slot_host, uint8_t *x_codes_host,
                                       uint8_t *x_scales_host, int32_t *slot_token_host);

/*   h_codes_host  uint8 [T*k, I/2]   requantised SwiGLU output of assignment a
 *                 ([T*k, I] for fp8xfp4)
 *   h_scales_host uint8 [T*k, I/32]  ([T*k, I/16] for nvf4xnvf4)
 *   h_scales_host uint8 [T*k, I/32]                                                   */
MXMOE_API moe_status moe_read_intermediate(const moe_dims *dims, const void *ws_dev,
                                           int32_t num_tokens, uint8_t *h_codes_host,
                                           uint8_t *h_scales_host);

/* Debug variant of the gate/up GEMM: writes the raw fp32 accumulators of every
 * assignment, de-interleaved, to gate_up_dev [T*k, 2I] (columns 0..I-1 gate,
 * I..2I-1 up) instead of running SwiGLU.  Runs after moe_pre_dispatch. */
MXMOE_API moe_status moe_debug_gate_up(const moe_dims *dims, const void *prepared_dev,
                                       void *ws_dev, size_t ws_bytes, float *gate_up_dev,
                                       int32_t num_tokens, void *stream);

/* Debug: exercises the bounded-wait failure path without any fault.  Launches one
 * block that waits, each time for at most limit_ns (1 us .. 1 s), on an mbarrier
 * nothing arrives at and on a workspace counter nothing increments -- the same
 * bounded waits the layer kernel uses.  Both give up; the block records a timeout
 * in the workspace flags and exits normally, so the context stays usable and the
 * next moe_check returns MOE_ERR_TIMEOUT. */
MXMOE_API moe_status moe_debug_wait_probe(void *ws_dev, int64_t limit_ns, void *stream);

/* ---- MXFP8 producer ----
 * SGLang PR #48424, section "DeepGEMM producers write FlashInfer's 128x4 scale
 * layout": a producer hands a downstream MXFP8 GEMM an FP8 pair, E4M3 values plus one
 * power-of-two (UE8M0) scale per 32 elements of a row, with the scales either packed
 * four to an int32 along K or written directly in the 4-D int32 layout
 * [ceil(rows/128), K/128, 32, 4], and padded rows' scales zeroed, so that the live
 * rows' scales are a prefix of a buffer sized for more rows.
 *
 * x   bf16 [rows, K] row-major, device, 16-byte aligned.
 * q   E4M3 codes [rows, K] row-major, device, 16-byte aligned (written).
 * sf  scales, device, 16-byte aligned, moe_mxfp8_scale_bytes(rows_cap, K, layout) bytes:
 *     MOE_SF_PACKED   int32 [rows_cap, K/128]; word j of a row holds groups 4j..4j+3
 *                     in its bytes 0..3; rows rows..rows_cap-1 are zeroed.
 *     MOE_SF_128X4    int32 [ceil(rows_cap/128), K/128, 32, 4]; the byte of (row r,
 *                     group s) sits at ((r/128)*(K/128) + s/4)*512 + (r%32)*16 +
 *                     ((r%128)/32)*4 + s%4; every row past `rows` is zeroed.
 * Each group's scale is 2^e, e the smallest integer with amax <= 448 * 2^e (clamped to
 * [-127, 127], amax = 0 gives -127), stored as the byte e + 127; each value is the
 * E4M3 value nearest to x * 2^-e, ties to the even code, sign kept.
 * 0 <= rows <= rows_cap <= 2^23, K a positive multiple of 128 (at most 65535 * 128 =
 * 8388480); inputs
 * finite.  Stream-ordered, no allocation, no synchronisation.  MOE_ERR_INVALID_ARG for
 * bad sizes, an unknown layout, or NULL / misaligned pointers. */
enum { MOE_SF_PACKED = 0, MOE_SF_128X4 = 1 };
MXMOE_API size_t moe_mxfp8_scale_bytes(int64_t rows_cap, int64_t K, int32_t sf_layout);
MXMOE_API moe_status moe_mxfp8_quantize(const void *x, int64_t rows, int64_t K, void *q,
                                        void *sf, int32_t sf_layout, int64_t rows_cap,
                                        void *stream);

/* FP4 tensor-core throughput probe (measurement only; the denominator of the
 * layer's compute roofline).  Launches `blocks` blocks of 128 threads on `stream`,
 * blocks_per_sm (1 or 2) of them resident per SM, each of which issues mma_count
 * (1 .. 2^20) block-scaled MXFP4 MMAs of shape M=128 x N=n x K=64 -- the layer's
 * instruction (kind::mxf4, UE8M0 scale per 32) -- on operands held in shared
 * memory, with no global-memory traffic.  n is 32, 64, 128 or 256 (256 only with
 * blocks_per_sm = 1).  The work is blocks * mma_count * 2*128*n*64 FLOP; the caller
 * times the launch with events on `stream`.  ws_dev is an initialised workspace
 * whose error flags receive MOE_ERR_TIMEOUT if the final wait exceeds 2 s (read by
 * moe_check).  Nothing is written to global memory otherwise.
 * Pages: "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE (W4A4)",
 * Appendix B (Compute SOL of the layer kernel). */
MXMOE_API moe_status moe_fp4_mma_probe(void *ws_dev, int32_t n, int32_t blocks_per_sm,
                                       int32_t blocks, int64_t mma_count, void *stream);

/* The probe's two-SM form: `pairs` clusters of two CTAs (one per SM), each pair's
 * leader issuing mma_count MXFP4 MMAs of shape M=256 x N=n x K=64 (tcgen05
 * cta_group::2: 128 of the 256 rows, and n/2 of B's rows, in each CTA's shared memory;
 * each CTA's accumulator rows in its own tensor memory).  n a multiple of 32 in
 * [32, 256]; 1 <= pairs <= 32768; 1 <= mma_count <= 2^20.  The work is
 * pairs * mma_count * 2*256*n*64 FLOP.  Errors and the timeout flag as for
 * moe_fp4_mma_probe.  Same page and section. */
MXMOE_API moe_status moe_fp4_mma_probe_pair(void *ws_dev, int32_t n, int32_t pairs,
                                            int64_t mma_count, void *stream);

/* ---- timing hooks ----
 * When enabled, moe_pre_dispatch and moe_forward record CUDA events around each
 * kernel they launch (on the launch stream).  moe_profile_read synchronises and
 * returns, per kernel name, the summed milliseconds and launch count since the
 * last reset.  names_out receives up to max_kernels static strings. */
MXMOE_API moe_status moe_profile_enable(int32_t on);
MXMOE_API int32_t moe_profile_read(const char **names_out, float *ms_out, int32_t *launches_out,
                                   int32_t max_kernels);
MXMOE_API void moe_profile_reset(void);

/* Number of SMs of the current device (what the persistent kernels size their
 * grids for); 0 if no device. */
MXMOE_API int32_t moe_device_sm_count(void);

/* ---- bucketing without any device allocation ----
 * The pages have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory where they route tokens: runtimes that plan every
 * device buffer ahead of time and forbid allocation afterwards, and latency-critical
 * threads that cannot afford cudaMalloc's implicit device-wide synchronisation.
 * Such a caller passes only its inputs and outputs.
 *
 * Runs the same bucketing kernel as moe_pre_dispatch on topk_ids_dev [T, k] and
 * topk_weights_dev [T, k] (T = num_tokens) and writes:
 *   counts_dev       int32 [E]    tokens routed to each expert
 *   assign_slot_dev  int32 [T*k]  row of assignment t*k+j in the expert-grouped order
 *                                 (experts' rows start at multiples of 128, tokens
 *                                 ascending inside an expert; -1 for ids outside [0, E))
 * -- the values moe_pre_dispatch stores in a workspace set to MOE_TILES_WIDE (see
 * moe_read_dispatch).
 * The kernel's other buffers live in a static device array of the library, about
 * 0.5 MiB, which every GPU that loads the library holds until the process exits.
 * Ids outside [0, E) are skipped: their assign_slot entry is -1 and they are not
 * counted, so the sum of counts_dev falls short of T*k by their number (no flag is
 * kept for them; moe_check does not see this call).
 * Limits: num_experts <= 256 and num_tokens * topk <= 8192; larger sizes return
 * MOE_ERR_INVALID_ARG without launching.  Only dims->num_experts, dims->topk
 * (1 <= topk <= min(num_experts, 32)) and dims->mma_type (a built type) are read;
 * hidden, inter and max_tokens are not used or checked.
 * The first call on a device looks up the array's device address (once per
 * device and context, with that device current; again after a device reset);
 * make that first call before any stream capture.  All calls share the array and it keeps the previous call's contents
 * (the error flags are cleared on every call); calls that overlap on the GPU --
 * on different streams or from different host threads -- race on it, so
 * serialise them.  Allocates nothing: no cudaMalloc, no cudaFree. */
MXMOE_API moe_status moe_bucket_noalloc(const moe_dims *dims, const int32_t *topk_ids_dev,
                                        const float *topk_weights_dev, int32_t num_tokens,
                                        int32_t *counts_dev, int32_t *assign_slot_dev,
                                        void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MXMOE_H */
