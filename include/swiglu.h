/*
 * swiglu.h - C ABI of libswiglu, the fused SwiGLU gated-MLP projection for
 * NVIDIA GB300 (sm_103a).
 *
 *   Y = SiLU(A x W1) (.) (A x W2)
 *
 * Operation: "Tile-Level Activation Overlap for Efficient LLM Inference"
 * (gist.science technical summary), section "Problem Statement": the gated MLP
 * multiplies the activations by two weight matrices and gates one product with
 * SiLU of the other. Section "Key Contributions" (tile-level fusion): the
 * intermediate Gate = A x W1 and Up = A x W2 are never written to memory; here
 * they live in fp32 tensor memory only.
 *
 * Types and layouts (all row-major, all bf16 unless stated):
 *   A   [M, K]  activations, K contiguous.
 *   W1  [K, N]  gate weight, N contiguous.   W2 [K, N] up weight, same layout.
 *   Wp  packed gate/up weight produced by swiglu_pack_weights (opaque to
 *       callers; layout stated at swiglu_pack_weights).
 *   Y   [M, N]  output, N contiguous.
 * Accumulation is fp32; SiLU(g) * u is evaluated in fp32 and rounded once to
 * bf16 (round to nearest even).
 *
 * Ownership: every buffer is allocated, owned and freed by the caller; pointers
 * are DEVICE pointers unless a parameter says "host". The library keeps one
 * small device status word per device (allocated on first use) and never
 * allocates on the forward path otherwise.
 *
 * Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL means
 * the legacy default stream). The return value reports argument errors and
 * launch errors only; device-side faults of the kind the kernels can detect
 * (a pipeline wait that ran past its time limit) are reported by
 * swiglu_check_device_status.
 *
 * Thread safety: calls may be made from several host threads; one-time set-up
 * per device is serialised internally.
 *
 * Environment (read once per process; for measurement and tuning, the
 * defaults are the measured choices):
 *   SWIGLU_PDL=0            launch without programmatic dependent launch.
 *   SWIGLU_SMALL_M_MAX=m    largest M for which the automatic choice always
 *                           takes the decode kernel (default 32).
 *   SWIGLU_L2_PREFETCH=n    packed tiles each decode CTA stages in L2 before
 *                           its grid-dependency wait (default: about 64 MB
 *                           over the grid, at most 16 per CTA; 4 in K-split
 *                           clusters).
 *   SWIGLU_L2_PREFETCH_LARGE=n  K slices each single-CTA kernel CTA stages in
 *                           L2 before its grid-dependency wait, for long K
 *                           loops (default: about 64 MB over the grid).
 *   SWIGLU_PAIR_GROUP_M=g   row tiles per group in the CTA-pair kernels' tile
 *                           order (default 16).
 *   SWIGLU_DOWN_CLUSTER=s, SWIGLU_DOWN_CLUSTERS=g  (both set) the decode
 *                           down-projection's K split with a workspace: g
 *                           clusters of s CTAs per output block, where they fit
 *                           (default: the measured rule of swiglu_down_forward_ws).
 *   SWIGLU_VERBOSE=1        swiglu_check_device_status prints the status record
 *                           (wait site, block, count) to stderr on a failure.
 */
#ifndef SWIGLU_H_
#define SWIGLU_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SWIGLU_API __attribute__((visibility("default")))
#else
#define SWIGLU_API
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* swiglu_stream_t;

typedef enum {
  SWIGLU_OK = 0,
  SWIGLU_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative or zero size, aliasing */
  SWIGLU_ERR_UNSUPPORTED = 2, /* K or N not a multiple of 8, size beyond limits, not sm_103 */
  SWIGLU_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
  SWIGLU_ERR_TIMEOUT = 4,     /* a kernel's pipeline wait exceeded its limit (device-side) */
  SWIGLU_ERR_NO_DEVICE = 5    /* no usable CUDA device / driver */
} swiglu_status_t;

/* Which kernel computes the forward pass. */
typedef enum {
  SWIGLU_VARIANT_AUTO = 0,    /* chosen from M (and the GPU's SM count) */
  SWIGLU_VARIANT_LARGE_M = 1, /* 128-token tiles of A, weight columns as the MMA N side */
  SWIGLU_VARIANT_SMALL_M = 2, /* weights as the MMA M side, tokens as N (M <= 256) */
  SWIGLU_VARIANT_LARGE_M_PAIR = 3, /* 256-token tiles on CTA pairs (tcgen05 cta_group::2) */
  SWIGLU_VARIANT_SEQUENTIAL = 4,   /* gate K loop, then up K loop with SiLU(gate) computed
                                      meanwhile: the pages' Kernel-1 schedule, for comparison */
  SWIGLU_VARIANT_SPLIT_K = 5,      /* 128 x 64 output tiles, each on a cluster of 2 CTAs that
                                      split K and sum their halves in shared memory (small
                                      single-wave problems) */
  SWIGLU_VARIANT_RESIDENT_PAIR = 6 /* 128 x 64 output tiles on CTA pairs (cta_group::2, M = 128)
                                      with every K slice loaded at once: K <= 896, bf16;
                                      UNSUPPORTED otherwise */
} swiglu_variant_t;

/*
 * Size in bytes of the packed weight for a K x N gate/up pair (infrastructure
 * of the boundary: no passage of the pages defines it; it sizes the buffer
 * swiglu_pack_weights fills):
 * 2 (matrices) * Np * Kp * 2 (bytes), Np = N rounded up to a multiple of 128,
 * Kp = K rounded up to a multiple of 64.
 * Returns 0 if K <= 0, N <= 0 or a size is beyond the limits below.
 */
SWIGLU_API size_t swiglu_packed_weight_bytes(int64_t K, int64_t N);

/*
 * Pack W1 and W2 into the layout the forward kernels stream from.
 *
 * The pages fuse the two weights into one K x 2N matrix so that matching Gate
 * and Up columns come out of one GEMM ("Tile-Level Activation Overlap for
 * Efficient LLM Inference", gist.science, section "Methodology / Kernel-2":
 * W_fused, even columns Gate, odd columns Up). This library interleaves blocks
 * of 128 columns instead of single columns, and stores each (column block,
 * 64-deep K slice) tile contiguously:
 *   Wp viewed as bf16 [Np/128][Kp/64][256][64]:
 *     Wp[j][b][i][t]       = W1[64b + t][128j + i]   (i < 128, gate)
 *     Wp[j][b][128 + i][t] = W2[64b + t][128j + i]   (i < 128, up)
 *   and 0 where 128j + i >= N or 64b + t >= K.
 * Each 32 KB tile is one load of the kernels' pipeline, one contiguous span.
 *
 * W1, W2: device, [K, N] bf16 row-major. Wpacked: device, at least
 * swiglu_packed_weight_bytes(K, N) bytes, must not overlap W1 or W2.
 * All three 16-byte aligned. Bit-exact copy; runs once per weight set.
 * Errors: INVALID_ARG (null, misaligned, K<=0, N<=0, overlap), UNSUPPORTED
 * (K or N not a multiple of 8, K or N above 2^21), NO_DEVICE, CUDA.
 */
SWIGLU_API swiglu_status_t swiglu_pack_weights(const void* W1, const void* W2, void* Wpacked,
                                               int64_t K, int64_t N, swiglu_stream_t stream);

/*
 * Y = SiLU(A x W1) (.) (A x W2), fused ("Tile-Level Activation Overlap for
 * Efficient LLM Inference", gist.science, sections "Problem Statement" and
 * "Methodology"): one pass over the packed weight; Gate and Up accumulate in
 * tensor memory, SiLU and the product run in the epilogue, Y is stored once.
 *
 * A: device [M, K] bf16. Wpacked: device, from swiglu_pack_weights with the
 * same K and N. Y: device [M, N] bf16, written in full, must not overlap A or
 * Wpacked. All 16-byte aligned.
 * M = 0 is a no-op returning OK.
 * Errors: INVALID_ARG (null or misaligned pointer, M < 0, K <= 0, N <= 0,
 * overlap), UNSUPPORTED (K or N not a multiple of 8; M above 2^31-1; K or N
 * above 2^21; device not sm_103), NO_DEVICE, CUDA (launch failure).
 */
SWIGLU_API swiglu_status_t swiglu_forward(const void* A, const void* Wpacked, void* Y,
                                          int64_t M, int64_t K, int64_t N,
                                          swiglu_stream_t stream);

/*
 * swiglu_forward with an explicit kernel choice (swiglu_variant_t); the
 * result is the same within rounding. SMALL_M requires M <= 256 (else
 * UNSUPPORTED).
 */
SWIGLU_API swiglu_status_t swiglu_forward_variant(const void* A, const void* Wpacked, void* Y,
                                                  int64_t M, int64_t K, int64_t N,
                                                  int variant, swiglu_stream_t stream);

/*
 * End-to-end form for callers whose activations live in host memory:
 * copies A_host -> A_dev, runs swiglu_forward(A_dev, Wpacked, Y_dev), copies
 * Y_dev -> Y_host, all enqueued on `stream` in that order (asynchronous: the
 * caller synchronises before reading Y_host). A_host and Y_host are HOST
 * pointers (page-locked memory gives asynchronous copies); A_dev and Y_dev are
 * caller-owned device staging buffers of 2*M*K and 2*M*N bytes.
 * Errors: as swiglu_forward, plus INVALID_ARG for null host pointers.
 */
SWIGLU_API swiglu_status_t swiglu_forward_from_host(const void* A_host, const void* Wpacked,
                                                    void* Y_host, void* A_dev, void* Y_dev,
                                                    int64_t M, int64_t K, int64_t N,
                                                    swiglu_stream_t stream);

/*
 * Infrastructure of the boundary (no passage of the pages defines it: the
 * pages describe no failure handling). Synchronises `stream`, then reads and
 * clears the current device's status word. Returns SWIGLU_ERR_TIMEOUT if any kernel since the last check gave up
 * on a pipeline wait (every wait in the kernels is bounded; the kernel then
 * stops cleanly and releases its resources), SWIGLU_ERR_CUDA if the stream
 * reports an error, SWIGLU_OK otherwise.
 */
SWIGLU_API swiglu_status_t swiglu_check_device_status(swiglu_stream_t stream);

/* Static, human-readable name of a status code (never NULL). Infrastructure of
 * the boundary; no passage of the pages defines it. */
SWIGLU_API const char* swiglu_status_string(swiglu_status_t status);

/*
 * Describes, as one line of text in `buf` (NUL-terminated, truncated to
 * `buflen`), the kernel and tiling swiglu_forward_variant would use for this
 * shape on the current device, e.g. "large_m bn=128 stages=4 tiles=4736
 * grid=152". Returns a status like swiglu_forward's argument checks.
 */
SWIGLU_API swiglu_status_t swiglu_plan_string(int64_t M, int64_t K, int64_t N, int variant,
                                              char* buf, size_t buflen);

/*
 * FP8 (E4M3) form of the op. The pages point out that quantisation raises
 * tensor-core throughput, which makes the memory-bound SwiGLU steps
 * relatively costlier ("Tile-Level Activation Overlap for Efficient LLM
 * Inference", gist.science, section "Problem Statement"); they give no
 * scaling scheme. Here each input is E4M3 values times one fp32 scale:
 *   A = scale_a * A8,  W1 = scale_w1 * W1_8,  W2 = scale_w2 * W2_8,
 *   Y = SiLU(A x W1) (.) (A x W2)   (bf16 output, fp32 accumulation; the
 *   products scale_a * scale_w1 and scale_a * scale_w2 are formed in fp32).
 * E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits, max 448, no infinity.
 *
 * Packed FP8 weight: as for bf16 but with 128 one-byte K values per slice,
 * viewed as bytes [Np/128][Kp/128][256][128], Kp = K rounded up to 128; size
 * 2 * Np * Kp bytes. swiglu_pack_weights_fp8 takes W1_8, W2_8 as [K, N]
 * E4M3 row-major device arrays. swiglu_forward_fp8 takes A8 [M, K] E4M3 and
 * writes Y [M, N] bf16; M <= 32 (or <= 64 on narrow N) uses the decode
 * kernel, larger M the CTA-pair kernel. Requirements and errors as the bf16 calls, plus K a multiple of 16
 * (UNSUPPORTED) and finite scales (INVALID_ARG).
 */
SWIGLU_API size_t swiglu_packed_weight_bytes_fp8(int64_t K, int64_t N);
SWIGLU_API swiglu_status_t swiglu_pack_weights_fp8(const void* W1, const void* W2, void* Wpacked,
                                                   int64_t K, int64_t N, swiglu_stream_t stream);
SWIGLU_API swiglu_status_t swiglu_forward_fp8(const void* A, const void* Wpacked, void* Y,
                                              int64_t M, int64_t K, int64_t N, float scale_a,
                                              float scale_w1, float scale_w2,
                                              swiglu_stream_t stream);
/*
 * swiglu_plan_string_fp8: the kernel and launch shape swiglu_forward_fp8
 * chooses for (M, K, N) on the current device, as text ("fp8 small_m ..." or
 * "fp8 large_m_pair ..."). buf NULL or buflen 0: INVALID_ARG; K not a
 * multiple of 16: UNSUPPORTED; no usable device: NO_DEVICE.
 */
SWIGLU_API swiglu_status_t swiglu_plan_string_fp8(int64_t M, int64_t K, int64_t N, char* buf,
                                                  size_t buflen);

/*
 * Block-scaled FP8 form of the op (MX: E4M3 values, one power-of-two scale per
 * 32 consecutive K values). As for the per-tensor form, the pages name FP8
 * only as the reason the SwiGLU steps weigh more once the GEMMs run faster
 * ("Tile-Level Activation Overlap for Efficient LLM Inference", gist.science,
 * section "Problem Statement"); they give no scaling scheme. Here:
 *   A[m][k]  = A8[m][k]  * 2^(SA[m][k/32] - 127)
 *   W1[k][n] = W1_8[k][n] * 2^(S1[k/32][n] - 127)      (W2 likewise with S2)
 *   Y = SiLU(A x W1) (.) (A x W2)   (bf16 output, fp32 accumulation)
 * Scales are UE8M0 bytes (value 2^(e - 127); 255 is NaN and must not occur);
 * A's scales run along its rows, W's down its columns. The tensor cores apply
 * both scales inside each MMA (tcgen05 kind::mxf8f6f4); no per-tensor factor.
 * K must be a multiple of 32 (else UNSUPPORTED); N a multiple of 8.
 *
 * Scale blocks: one 512-byte block holds the scales of 128 rows x 4 groups
 * (128 K values); row r, group g at byte (r % 32) * 16 + (r / 32) * 4 + g.
 *
 * swiglu_packed_weight_bytes_mxfp8(K, N): bytes of the packed weight: the
 *   E4M3 values exactly as swiglu_pack_weights_fp8 lays them out (2 * Np * Kp
 *   bytes, Kp = K rounded up to 128), followed by 1024 bytes per packed tile
 *   (column block j, K slice b, same tile order): W1's scale block for columns
 *   128j .. 128j+127 and groups 4b .. 4b+3, then W2's; 127 where no value is.
 * swiglu_pack_weights_mxfp8: W1_8, W2_8 [K, N] E4M3 and S1, S2 [K/32, N]
 *   UE8M0, row-major device arrays, into Wpacked (device, 16-byte aligned, of
 *   swiglu_packed_weight_bytes_mxfp8 bytes, overlapping none of them).
 * swiglu_act_scale_bytes_mxfp8(M, K): bytes of A's scales in blocks:
 *   ceil(M/128) x ceil(K/128) blocks of 512 bytes, row-block major.
 * swiglu_pack_act_scales_mxfp8: SA [M, K/32] UE8M0 row-major (device) into
 *   that block layout (SAtiled, device, 16-byte aligned); 127 where no row or
 *   group is. A producer of quantised activations may write the block layout
 *   directly instead.
 * swiglu_forward_mxfp8: A8 [M, K] E4M3 (device), SAtiled (from the call
 *   above), Wpacked (from swiglu_pack_weights_mxfp8 with the same K, N), Y
 *   [M, N] bf16 (device, written in full, overlapping no input). All 16-byte
 *   aligned. M = 0 is a no-op. Few tokens (the FP8 decode rule, at most 128)
 *   run the decode kernel, others the CTA-pair kernel.
 * swiglu_plan_string_mxfp8: the kernel and launch shape swiglu_forward_mxfp8
 *   chooses for (M, K, N) on the current device, as text ("mxfp8 ...").
 * Errors as the bf16 calls.
 */
SWIGLU_API size_t swiglu_packed_weight_bytes_mxfp8(int64_t K, int64_t N);
SWIGLU_API swiglu_status_t swiglu_pack_weights_mxfp8(const void* W1, const void* S1,
                                                     const void* W2, const void* S2,
                                                     void* Wpacked, int64_t K, int64_t N,
                                                     swiglu_stream_t stream);
SWIGLU_API size_t swiglu_act_scale_bytes_mxfp8(int64_t M, int64_t K);
SWIGLU_API swiglu_status_t swiglu_pack_act_scales_mxfp8(const void* SA, void* SAtiled, int64_t M,
                                                        int64_t K, swiglu_stream_t stream);
SWIGLU_API swiglu_status_t swiglu_forward_mxfp8(const void* A, const void* SAtiled,
                                                const void* Wpacked, void* Y, int64_t M,
                                                int64_t K, int64_t N, swiglu_stream_t stream);
SWIGLU_API swiglu_status_t swiglu_plan_string_mxfp8(int64_t M, int64_t K, int64_t N, char* buf,
                                                   size_t buflen);

/*
 * The gated MLP's down-projection, the step after Y in the models the pages
 * evaluate ("Tile-Level Activation Overlap for Efficient LLM Inference",
 * gist.science, section "Problem Statement": the SwiGLU gated MLP; the pages
 * do not describe this step further):
 *   Out [M, H] = Y [M, N] x W3 [N, H] + R [M, H]     (bf16, fp32 accumulation)
 * Y is the fused forward's output (N = the intermediate size), H the hidden
 * size, R the block's residual input (NULL: none). Out may be R itself
 * (in-place residual add); any other overlap is INVALID_ARG.
 * Packed W3: tiles of 256 output columns x 64 K values, viewed as bf16
 * [Hp/256][Np/64][256][64] with Wp[j][b][i][t] = W3[64b + t][256j + i], zero
 * past the edges (Hp, Np = H, N rounded up to 256, 64); size
 * swiglu_down_packed_bytes(N, H). M <= 64 (or M <= 128 with few 256-column
 * output blocks) runs the decode kernel, with K split over clusters when H is
 * narrow; larger M the CTA-pair kernel. N and H multiples of 8; errors as
 * swiglu_forward.
 */
SWIGLU_API size_t swiglu_down_packed_bytes(int64_t N, int64_t H);
SWIGLU_API swiglu_status_t swiglu_pack_down_weights(const void* W3, void* W3packed, int64_t N,
                                                    int64_t H, swiglu_stream_t stream);
SWIGLU_API swiglu_status_t swiglu_down_forward(const void* Y, const void* W3packed, const void* R,
                                               void* Out, int64_t M, int64_t N, int64_t H,
                                               swiglu_stream_t stream);

/*
 * swiglu_down_plan_string: the kernel and launch shape swiglu_down_forward
 * chooses for (M, N, H) on the current device, as text ("down small_m ..." or
 * "down large_m_pair ..."). buf NULL or buflen 0: INVALID_ARG; no usable
 * device: NO_DEVICE; bad shape: as swiglu_down_forward.
 */
SWIGLU_API swiglu_status_t swiglu_down_plan_string(int64_t M, int64_t N, int64_t H, char* buf,
                                                   size_t buflen);

/*
 * Down-projection with a caller workspace. With few 256-column output blocks
 * and few tokens (the decode kernel), one cluster of CTAs per block leaves
 * most SMs idle while the weight stream is the whole cost; with a workspace
 * the block's K range is also split across several clusters, which write fp32
 * partial sums to the workspace, and the last cluster of each block to finish
 * adds them in cluster order (so results do not depend on timing) and writes
 * Out. Same result rule as swiglu_down_forward; the two may differ in the
 * last bits of the fp32 sums (a different summation order) before rounding.
 *
 * swiglu_down_workspace_bytes(M, N, H): bytes that call needs for (M, N, H) on
 *   the current device; 0 when its plan does not split K across clusters (or
 *   on a bad shape or no usable device).
 * swiglu_down_forward_ws: as swiglu_down_forward, plus `workspace` (device,
 *   16-byte aligned, overlapping no other argument) of `workspace_bytes`.
 *   workspace NULL: exactly swiglu_down_forward. Otherwise, if the plan needs
 *   a workspace, workspace_bytes below swiglu_down_workspace_bytes or a bad
 *   pointer: INVALID_ARG. Contents: the first bytes hold arrival counters that
 *   must be zero when a call's kernel starts; the caller zero-fills the
 *   workspace once before its first use, and every call's kernel leaves them
 *   at zero again when it ends (also when a pipeline wait timed out), so a
 *   workspace serves any number of calls in stream order. Calls that may run
 *   at the same time (different streams) need separate workspaces. The
 *   library never allocates it.
 * swiglu_down_plan_string_ws: the plan swiglu_down_forward_ws takes with a
 *   workspace ("clusters=g": K split across g clusters per block).
 */
SWIGLU_API size_t swiglu_down_workspace_bytes(int64_t M, int64_t N, int64_t H);
SWIGLU_API swiglu_status_t swiglu_down_forward_ws(const void* Y, const void* W3packed,
                                                  const void* R, void* Out, int64_t M, int64_t N,
                                                  int64_t H, void* workspace,
                                                  size_t workspace_bytes, swiglu_stream_t stream);
SWIGLU_API swiglu_status_t swiglu_down_plan_string_ws(int64_t M, int64_t N, int64_t H, char* buf,
                                                      size_t buflen);

/*
 * Allocation-free forward for callers that cannot call cudaMalloc: serving
 * runtimes that reserve all device memory for their own pools up front (a
 * library allocation would fail, or would fragment memory the runtime plans
 * to the byte), and hosts that forbid allocation once start-up is over. The
 * other forward entry points allocate one small status record per device on
 * first use; this one runs the decode (small-M) kernel with that record in a
 * file-scope static device array of 256 bytes instead, held by every GPU that
 * loads the library until the process exits. No passage of the method covers it:
 * this is a deployment variant, not part of the method.
 *
 * Same arguments and result as swiglu_forward, for M <= 256 (larger M:
 * UNSUPPORTED). The launch shape does not depend on the device: one CTA per
 * 128-column block holding all M tokens (no K split over clusters, no token
 * groups), so it can differ from swiglu_forward's for M > 32 or narrow N.
 * The caller passes every input and output; the library allocates nothing
 * (no cudaMalloc, cudaFree or allocating library call).
 * Each call clears the shared status record on `stream` before the kernel;
 * if `status_out` (HOST, 4 x uint32, may be NULL) is given, the record is
 * copied there after the kernel, on `stream`: status_out[0] is 0, or 4
 * (SWIGLU_ERR_TIMEOUT) if a pipeline wait gave up; read it after the stream
 * synchronises (page-locked memory keeps the copy asynchronous; pageable
 * memory makes the call wait for the kernel).
 * The first call on a device does a one-time set-up (kernel attributes and the
 * array's device address, both host-side CUDA runtime queries).
 * Calls whose kernels overlap on the GPU (several streams) share the record
 * and race on it; serialise them to get a meaningful status.
 */
SWIGLU_API swiglu_status_t swiglu_forward_noalloc(const void* A, const void* Wpacked, void* Y,
                                                  int64_t M, int64_t K, int64_t N,
                                                  uint32_t* status_out, swiglu_stream_t stream);

/*
 * Testing hook for the failure path: while `enable` is non-zero, the next
 * forward launches skip one pipeline-stage fill, so a wait inside the kernel
 * runs out after `timeout_ms` milliseconds (default 1000) and the kernel exits
 * with SWIGLU_ERR_TIMEOUT recorded. `timeout_ms` = 0 keeps the current limit.
 */
SWIGLU_API void swiglu_testing_inject_stall(int enable, uint32_t timeout_ms);

/*
 * Testing counter of the CTA-pair kernel's tile-round pacing (bf16 gate/up,
 * K >= 8192: each pair waits, bounded, for every pair of the launch to have
 * issued the loads of the tile two rounds back; a wait that runs out only
 * turns pacing off for the rest of that launch). Writes to `*count` (HOST)
 * the number of such waits that ran out on the current device since the
 * library was loaded. Synchronous with the device (reads a device counter).
 * No passage of the method defines it: it is test infrastructure of the
 * boundary. Errors: INVALID_ARG (count NULL), NO_DEVICE, CUDA.
 */
SWIGLU_API swiglu_status_t swiglu_testing_pace_run_out(uint64_t* count);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_H_ */
