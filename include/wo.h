/*
 * wo.h -- C ABI of libwo, the weight-only quantized fpA.intB GEMM for GB300
 * (sm_103a):
 *
 *     C[m, n] = A[m, k] . dequant(B)^T + bias[n]
 *
 * A holds fp16 or bf16 activations; B holds integer weight codes of the
 * output channels (n) along the reduction dimension (k):
 *   - bits 8 (A16W8): uint8 codes 0..255, w = (q - 128) * scale[n], one scale
 *     per output channel ("acext User Guide (v1.7)" 1.3.1 Int8 Weight-only;
 *     "[Misc][Kernel]: Add GPTQAllSpark Quantization": group_size -1, no
 *     act-order);
 *   - bits 4 (W4A16): two codes per byte, w = (q - 8) * scale[n][g] +
 *     zero[n][g] per group g of group_size codes along k (acext 1.3.3 Int4
 *     Groupwise; vLLM-Omni "cpu_int4.py" module docstring).
 *
 * The calls follow the runner convention of acext 1.2.1 (fpAintB GEMM):
 * the caller owns every buffer, including the workspace whose size the
 * library reports, and passes an explicit stream; work is stream-ordered and
 * asynchronous.  No entry point allocates or frees device memory.
 *
 * Conventions for every call below:
 *   - Pointers named for tensors are DEVICE pointers owned by the caller and
 *     must stay valid until the stream work completes.  A, B, C, out and the
 *     packed buffers must be 16-byte aligned, the workspace 256-byte aligned,
 *     scales, zeros and bias 2-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Argument checks happen before any launch; on an error no work is
 *     enqueued.  WO_ERR_CUDA reports a launch failure (cudaGetLastError).
 *   - fp16/bf16 tensors are 16-bit IEEE binary16 / bfloat16 values.
 *   - Every 16-bit output is rounded to nearest even once, from fp32.
 */
#ifndef WO_H
#define WO_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define WO_API __attribute__((visibility("default")))
#else
#define WO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WO_OK = 0,
    WO_ERR_INVALID_ARG = 1, /* a null/misaligned pointer, a bad size or enum */
    WO_ERR_UNSUPPORTED = 2, /* a valid combination this library does not run */
    WO_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    WO_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    WO_ERR_TIMEOUT = 5,     /* a kernel gave up a bounded wait (see wo_check_workspace) */
    WO_ERR_BOUNDS = 6       /* debug build: an index check failed (see wo_debug_bounds) */
} wo_status;

typedef enum { WO_F16 = 0, WO_BF16 = 1 } wo_dtype;

/* Human-readable name of a status.  Never NULL. */
WO_API const char* wo_status_string(wo_status s);

/*
 * Bytes of the packed weight buffer for an [n, k] code matrix: n*k (bits 8)
 * or n*k/2 (bits 4).  0 for invalid arguments.  Packing keeps the byte count.
 */
WO_API size_t wo_packed_bytes(int n, int k, int bits);

/*
 * Offline repack of row-major codes into the tile-interleaved layout every
 * GEMM kernel here reads (the analogue of acext's
 * preprocess_weights_for_mixed_gemm, 1.3.1-1.3.3, run once at load).
 *   B_rowmajor: bits 8: uint8 [n, k]; bits 4: uint8 [n, k/2] with byte j of a
 *               row = code 2j | code 2j+1 << 4 (cpu_int4.py docstring).
 *   B_packed:   wo_packed_bytes(n, k, bits) bytes; must not overlap B_rowmajor.
 * Layout of B_packed: 512-byte tiles of 16 output channels by 32 (bits 8) or
 * 64 (bits 4) codes, tiles ordered by channel block then by k; inside a tile
 * lane L (0..31) owns bytes 16L..16L+15, which hold exactly the codes of the
 * m16n8k16 A-operand fragments of lane L for the tile's k-steps.
 * Requires n % 64 == 0, k % 64 == 0, k > 0, n > 0; bits in {4, 8}.
 * Bit-exact and invertible: wo_unpack(wo_pack(x)) == x.
 */
WO_API wo_status wo_pack(const uint8_t* B_rowmajor, uint8_t* B_packed, int n, int k, int bits,
                  void* stream);

/* Inverse of wo_pack (same arguments, same requirements). */
WO_API wo_status wo_unpack(const uint8_t* B_packed, uint8_t* B_rowmajor, int n, int k, int bits,
                    void* stream);

/*
 * Workspace bytes wo_gemm needs for this problem (acext 1.2.1
 * getWorkspaceSize).  May be 0.  The workspace must be zero-filled before its
 * first use (cudaMemset); every call leaves it ready for the next one.  Calls
 * that share a workspace must be ordered on one stream.
 */
WO_API size_t wo_workspace_size(int m, int n, int k, int group_size, int bits);

/*
 * The weight-only GEMM (acext 1.2.1 gemm(A, B, weight_scales,
 * weight_zero_points, biases, C, m, n, k, group_size, ...)).
 *   A:        act_dtype [m, k], row-major.
 *   B_packed: output of wo_pack for (n, k, bits).
 *   scales:   act_dtype; per channel ([n]) when group_size is -1 or k,
 *             otherwise [n, k/group_size].
 *   zeros:    same shape and dtype as scales, or NULL (= 0).  bits 4 only.
 *   bias:     act_dtype [n] or NULL.
 *   C:        act_dtype [m, n], row-major; must not overlap the inputs.
 *   bits 8: group_size -1 or k (per channel), zeros NULL.
 *   bits 4: group_size 64 or 128 (a multiple of 64 dividing k), or -1/k.
 * Requires n % 64 == 0, k % 64 == 0 and k > 0; m == 0 or n == 0 is a no-op.
 * The kernel is chosen by m: for 4-bit weights at decode-sized m (1..16)
 * a persistent weight-streaming kernel where the cluster-split one would
 * need more than one resident wave of CTAs, as for a wide lm_head
 * (group-wise weights also need 16-byte aligned scales and
 * zeros and k / group_size a multiple of 8); for 8-bit weights at 17..64
 * rows (n % 128 == 0) a tcgen05 kernel with the weights as the MMA's rows
 * while n / 128 is at most the SM count, the m >= 65 tensor-core kernel for
 * wider n; otherwise up to m = 64 a cluster-split weight-streaming kernel,
 * and a tcgen05 tensor-core kernel for larger m (wo_gemm_plan reports the
 * choice).  Results are deterministic: identical inputs give
 * bit-identical C.
 * Ordering: the small-m kernel uses programmatic dependent launch.  It may
 * start reading B_packed, scales, zeros and bias while the previous
 * operation on the stream is still running, so those must not be written by
 * the immediately preceding kernel on the stream (weights packed at load
 * time, with any synchronisation in between, are fine).  A is read and C
 * written only after the previous operation has completed, as usual.
 */
WO_API wo_status wo_gemm(const void* A, const uint8_t* B_packed, const void* scales,
                  const void* zeros, const void* bias, void* C, int m, int n, int k,
                  int group_size, int bits, wo_dtype act_dtype, void* workspace,
                  size_t workspace_bytes, void* stream);

/*
 * The configuration wo_gemm runs for a problem (the counterpart of acext
 * 1.2.1's getChosenConfig, which returns the kernel configuration a runner
 * will use; here the choice is a static plan, reported, not passed in).
 * Pure host code: no CUDA call beyond reading the device's SM count (152
 * when no device is visible).
 */
typedef enum {
    WO_KERNEL_STREAM = 0,            /* cluster-split weight streaming (m <= 64) */
    WO_KERNEL_TENSOR_CORE = 1,       /* tcgen05 tensor cores (m >= 65) */
    WO_KERNEL_STREAM_PERSISTENT = 2, /* persistent weight streaming (4-bit, m <= 16) */
    WO_KERNEL_TENSOR_CORE_SWAP_AB = 3 /* tcgen05 with the weights as the MMA's rows
                                        (8-bit, 17 <= m <= 64) */
} wo_kernel;

typedef struct {
    wo_kernel kernel;      /* which kernel family runs */
    int tile_m;            /* rows of C per CTA tile (streaming: m) */
    int tile_n;            /* output channels per CTA tile (persistent: per strip) */
    int k_splits;          /* CTAs of one cluster (streaming), units per tile along k
                              (tensor cores, swap AB), or the most pieces one strip's k
                              range is cut into across CTAs (persistent) */
    int ctas;              /* CTAs launched */
    int stages;            /* streaming: shared-memory ring stages per CTA; else 0 */
    size_t workspace_bytes; /* == wo_workspace_size */
} wo_gemm_plan_t;

/*
 * Fills *plan for wo_gemm(m, n, k, group_size, bits, act_dtype).  Same
 * argument rules as wo_gemm; WO_ERR_INVALID_ARG for a NULL plan; m == 0 or
 * n == 0 gives a plan with ctas == 0.
 */
WO_API wo_status wo_gemm_plan(int m, int n, int k, int group_size, int bits, wo_dtype act_dtype,
                              wo_gemm_plan_t* plan);

/*
 * GPTQ act-order checkpoints ("[Misc][Kernel]: Add GPTQAllSpark
 * Quantization": the desc_act / has_g_idx case its kernel leaves out).  The
 * quantiser visited the input channels in its own order, so input channel c
 * belongs to group g_idx[c] rather than c / group_size:
 *     C[m, n] = sum_c A[m, c] * ((q[n][c] - 8) * scale[n][g_idx[c]]
 *                                + zero[n][g_idx[c]]) + bias[n].
 * A sum over k does not depend on the order of its terms, so sorting the
 * channels by group turns this into the ordinary group-wise GEMM: the codes
 * are packed in sorted order once (wo_pack_act_order), and each call gathers
 * A's columns into the same order before the group-wise kernels run
 * (wo_gemm_act_order).  scales and zeros stay [n, k/group_size], indexed by
 * group number; A, B_rowmajor and C keep the checkpoint's channel order.
 */

/*
 * The channel order that sorts a group index, on the HOST.
 *   g_idx: HOST int32 [k], the group of each input channel, 0 <= g_idx[c] <
 *          k / group_size (group_size -1 or k: one group, all entries 0).
 *   perm:  HOST int32 [k] output: perm[j] = the j-th channel in order of
 *          (g_idx[c], c), so positions [b*group_size, (b+1)*group_size) hold
 *          the channels of group b.
 * WO_ERR_INVALID_ARG for a null pointer, k <= 0, a group_size that does not
 * divide k or an entry outside [0, k/group_size); WO_ERR_UNSUPPORTED when the
 * groups are not all exactly group_size channels (GPTQ's are).  Pure host
 * code: no CUDA call.
 */
WO_API wo_status wo_act_order_perm(const int32_t* g_idx, int k, int group_size, int32_t* perm);

/*
 * wo_pack with the input channels reordered: packed column j holds
 * row-major column perm[j].  perm is a DEVICE int32 [k] (4-byte aligned),
 * the output of wo_act_order_perm copied to the device; an entry outside
 * [0, k) packs code 0 (no out-of-bounds read).  Other arguments and
 * requirements as wo_pack.  wo_unpack of the result gives the row-major
 * codes with columns in the order perm.
 */
WO_API wo_status wo_pack_act_order(const uint8_t* B_rowmajor, uint8_t* B_packed,
                                   const int32_t* perm, int n, int k, int bits, void* stream);

/*
 * Workspace bytes of wo_gemm_act_order: the wo_gemm workspace of the same
 * problem, at least its shared header and split-K counter area
 * (256 + 65536 bytes), rounded up to 256, followed by an act_dtype [m, k]
 * copy of A in sorted channel order.  0 for invalid arguments or m == 0 or
 * n == 0.  The zero-fill rule of wo_gemm's workspace applies to the whole
 * buffer, and one buffer may serve wo_gemm and wo_gemm_act_order calls in
 * turn (on one stream).
 */
WO_API size_t wo_act_order_workspace_size(int m, int n, int k, int group_size, int bits);

/*
 * The act-order GEMM above.
 *   A:        act_dtype [m, k] in the checkpoint's channel order.
 *   B_packed: output of wo_pack_act_order with the same perm.
 *   perm:     DEVICE int32 [k], 16-byte aligned, from wo_act_order_perm; an
 *             entry outside [0, k) reads A as 0.
 *   other arguments, requirements and the ordering rule: as wo_gemm, with
 *   the workspace sized by wo_act_order_workspace_size.
 * Runs a column gather of A into the workspace (a programmatic dependent
 * launch: it reads perm before the previous operation on the stream
 * completes, A after), then the wo_gemm kernels on the gathered copy.
 */
WO_API wo_status wo_gemm_act_order(const void* A, const uint8_t* B_packed, const int32_t* perm,
                                   const void* scales, const void* zeros, const void* bias,
                                   void* C, int m, int n, int k, int group_size, int bits,
                                   wo_dtype act_dtype, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * Rows of a quantised embedding (vocab) table, dequantised (vLLM-Omni
 * "cpu_int4.py", CPUInt4EmbeddingMethod.embedding: the rows of the token ids,
 * w = (q - offset) * scale (+ zero) in fp32, rounded once to the activation
 * dtype).  The table is the same packed weight wo_gemm reads as [n, k] =
 * [vocab, hidden] (tied lm_head and embedding share one copy): rows are read
 * straight from the packed tiles.
 *   ids:      int32 [T] device array of token ids; an id outside [0, vocab)
 *             gives a row of zeros.
 *   B_packed: output of wo_pack for (vocab, hidden, bits).
 *   scales, zeros, group_size, bits: as for wo_gemm (n = vocab, k = hidden).
 *   out:      act_dtype [T, hidden], row-major.
 * Requires vocab % 64 == 0, hidden % 64 == 0; T == 0 is a no-op.  Pointers:
 * ids 4-byte, B_packed and out 16-byte, scales and zeros 2-byte aligned.
 * Bit-identical to rounding the oracle's fp32 dequantised rows.
 */
WO_API wo_status wo_embed(const int32_t* ids, int T, const uint8_t* B_packed, const void* scales,
                          const void* zeros, void* out, int vocab, int hidden, int group_size,
                          int bits, wo_dtype act_dtype, void* stream);

/*
 * Workspace bytes for wo_moe_ffn with T tokens, the given sizes and top-k.
 * Same zero-fill rule as wo_workspace_size.
 */
WO_API size_t wo_moe_workspace_size(int T, int hidden, int inter, int experts, int topk);

/*
 * Grouped weight-only MoE FFN (acext 1.2.3 MoE GEMM runner: gating output,
 * top-k experts per row, fc1 with a gated activation, fc2, routing-weighted
 * combine):
 *   ids[t], p[t] = top-k of gating_logits[t] (ties to the lower expert id),
 *                  p = softmax probabilities over all experts of the chosen
 *                  ids (renormalised to sum 1 when renormalize != 0);
 *   for each chosen expert e: [g | u] = A[t] . dequant(fc1_e)^T (2*inter),
 *                  h = round(silu(g) * u), y = h . dequant(fc2_e)^T;
 *   out[t] = round(sum_j p[t][j] * y_j).
 *   A:             act_dtype [T, hidden].
 *   gating_logits: fp32 [T, experts].
 *   fc1_packed:    experts consecutive wo_pack outputs of [2*inter, hidden]
 *                  bits-8 codes; fc1_scales act_dtype [experts, 2*inter].
 *   fc2_packed:    experts consecutive wo_pack outputs of [hidden, inter];
 *                  fc2_scales act_dtype [experts, hidden].
 *   out:           act_dtype [T, hidden].
 * Requires hidden % 64 == 0, inter % 64 == 0, 1 <= topk <= experts <= 1024.
 */
WO_API wo_status wo_moe_ffn(const void* A, const float* gating_logits, const uint8_t* fc1_packed,
                     const void* fc1_scales, const uint8_t* fc2_packed,
                     const void* fc2_scales, void* out, int T, int hidden, int inter,
                     int experts, int topk, int renormalize, wo_dtype act_dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * wo_gemm without a workspace, for callers that cannot allocate device
 * memory themselves (for example a plugin running inside an engine that owns
 * all device memory through its own pool, or latency-critical code that must
 * not call cudaMalloc, which can synchronise the device).  The pages have no
 * counterpart: their runners always take a caller-allocated workspace.
 *   Arguments as for wo_gemm, minus the workspace.  Always runs the
 *   tensor-core kernel, whatever m is.
 *   Scratch: a 24.06 MiB array in the library's device memory, held on every
 *   GPU that loads the library until the process exits.  8-bit weights need
 *   none of it.  4-bit weights need, each rounded up to 256 bytes, within
 *   24 MiB in all: n*(k/group_size)*4 bytes of pre-scaled scale and zero
 *   pairs, n*2 bytes of column scales and, with bf16 activations, the fp16
 *   copy of A (m*k*2 bytes) and its row scales (m*4 bytes) -- e.g. m*k up
 *   to about 12 million; larger problems return WO_ERR_WORKSPACE with
 *   nothing enqueued.
 *   Every call looks up the array's address in the caller's current CUDA
 *   context (a host-side lookup), so another context, or a primary context
 *   recreated by cudaDeviceReset, uses its own copy.  The first call in a
 *   context zeroes that copy's error word (a blocking cudaMemset), so make
 *   that first call before any stream capture.  The call allocates and frees
 *   nothing.  Every call shares the array: calls whose kernels overlap on the
 *   GPU (unordered streams) race on it.  A kernel that gives up a bounded
 *   wait records it in the array's error word: wo_noalloc_check reads it.
 */
WO_API wo_status wo_gemm_tc_noalloc(const void* A, const uint8_t* B_packed, const void* scales,
                                    const void* zeros, const void* bias, void* C, int m, int n,
                                    int k, int group_size, int bits, wo_dtype act_dtype,
                                    void* stream);

/*
 * The failure report of wo_gemm_tc_noalloc (no counterpart on the pages):
 * synchronises `stream`, then reads and clears the error word of the
 * built-in scratch of the current context.  Returns WO_OK, WO_ERR_TIMEOUT
 * (a kernel gave up a bounded wait since the last check), or WO_ERR_CUDA.
 */
WO_API wo_status wo_noalloc_check(void* stream);

/*
 * Synchronises `stream`, then reads and clears the error word a kernel may
 * have left in `workspace` (a tensor-core kernel that gave up a bounded wait
 * writes it instead of hanging).  Returns WO_OK, WO_ERR_TIMEOUT, or
 * WO_ERR_CUDA when the stream reported an error.  After WO_ERR_TIMEOUT the
 * workspace's counters may not be back at zero: zero-fill the workspace
 * again before its next use.
 */
WO_API wo_status wo_check_workspace(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Index checks of the debug build (no counterpart on the pages; a stand-in
 * for a memory checker, which this project's GPUs do not offer).  A library
 * compiled with -DWO_DEBUG_BOUNDS=1 checks every global index its kernels
 * compute (plain loads and stores; TMA boxes are clipped by the hardware)
 * against the extent of the buffer; a failed check skips the access and
 * records a site code (0x100-0x7ff, the kernel family in the high digit) in
 * a device word instead of faulting.  This call waits for the device, then
 * reads and clears those words: WO_OK if no check failed since the last
 * call, WO_ERR_BOUNDS with the first failed check's site in *site (may be
 * NULL); WO_ERR_UNSUPPORTED from a library built without the checks;
 * WO_ERR_CUDA if the device reported an error.
 */
WO_API wo_status wo_debug_bounds(unsigned* site);

/*
 * Self-test of the failure path (no counterpart on the pages): launches one
 * CTA whose thread waits on an mbarrier that nothing ever arrives on, with
 * the same bounded wait the kernels use but a limit of `limit_us`
 * microseconds (1..1000000).  The wait runs out, the CTA records its error
 * code in `workspace`'s error word and exits; the GPU is not left hanging
 * and the context stays usable.  wo_check_workspace then returns
 * WO_ERR_TIMEOUT (and clears the word).  workspace: at least 256 bytes,
 * 256-byte aligned.
 */
WO_API wo_status wo_selftest_wait_timeout(void* workspace, size_t workspace_bytes, unsigned limit_us,
                                          void* stream);

/*
 * wo_selftest_wait_timeout on the built-in scratch of wo_gemm_tc_noalloc
 * (no counterpart on the pages): the bounded wait runs out after `limit_us`
 * microseconds (1..1000000) and records its code in that scratch's error
 * word, which wo_noalloc_check then reports as WO_ERR_TIMEOUT.
 */
WO_API wo_status wo_noalloc_selftest_wait_timeout(unsigned limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WO_H */
