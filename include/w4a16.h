/*
 * w4a16.h -- C ABI of libw4a16.so: a W4A16 group-quantized linear layer for
 * NVIDIA B300 (sm_103a).
 *
 * The layer computes y = x . W_hat^T, where W_hat[n][k] = (q[n][k] - z) * s:
 * 4-bit codes q, one fp16 scale s and one 4-bit zero point z per (row, group)
 * of `group_size` input columns, fp16 activations x and outputs y, fp32
 * accumulation. The same entry points take 8-bit codes (W8A16, the wider
 * choice weighed in "AWQ + GPTQ Quantization, in depth", section "4-bit bigger
 * or 8-bit smaller") and 3-bit codes (W3A16; 3 and 8 bits are the other widths
 * named in "How do GPTQ and AWQ differ ...", section "The shared setting"). The format follows "AWQ + GPTQ Quantization, in depth",
 * section "What W4A16 buys and why decoding gets faster" (packed 4-bit weights
 * expanded to 16 bits in registers with the group's scale and zero point; one
 * scale per group of 128 neighbouring input columns of a row) and "LLM
 * Quantization: A Deep Dive into GPTQ, AWQ, and Post-Training Quantization",
 * section "The Math of Quantization" (q = round(x/S) + Z, x ~ (q - Z) * S).
 * The knobs -- bits, group_size, symmetric/zero point, act order (desc_act,
 * g_idx) -- are those of the Q&A page "How do GPTQ and AWQ differ when
 * quantizing Llama weights to 4 bits?", section "GPTQ: quantize then
 * compensate".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Ownership: the caller allocates and frees every buffer. The library
 *   allocates no memory and keeps no state besides a per-device cache of
 *   device attributes.
 * - Pointers are device pointers unless the argument says "host".
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) except where noted, and is reentrant.
 * - Arguments are validated on the host before anything is launched; on any
 *   error nothing is launched and nothing is written.
 * - Unsupported combinations return W4A16_ERR_UNSUPPORTED; there is no slower
 *   fallback path (a silent fallback is the failure mode named in "AWQ + GPTQ
 *   Quantization, in depth", section "Failure modes": "Kernel fallback").
 * - A failed CUDA launch returns W4A16_ERR_CUDA; w4a16_last_cuda_error() then
 *   gives the cudaError_t (per calling thread). Nothing aborts, prints or traps.
 * - Results are deterministic for a given (format, M, device): fixed reduction
 *   order, no floating-point atomics.
 *
 * Element types: fp16 values are passed as uint16_t bit patterns (IEEE binary16).
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* w4a16_stream_t;

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1,     /* NULL pointer, bad size, M out of range, bad g_idx */
  W4A16_ERR_UNSUPPORTED = 2,     /* valid but not implemented (bits not 3, 4 or 8, group size, ...) */
  W4A16_ERR_MISALIGNED = 3,      /* a pointer is not aligned as documented */
  W4A16_ERR_BUFFER_TOO_SMALL = 4,/* packed_bytes or workspace_bytes below the requirement */
  W4A16_ERR_CUDA = 5             /* a CUDA call failed; see w4a16_last_cuda_error() */
} w4a16_status;

/*
 * Quantization format of one linear layer (out features N x in features K).
 *   bits        3, 4 or 8 (b below; codes 0 .. 2^b - 1).
 *   group_size  32, 64 or 128; K must be a multiple of it (G = K / group_size
 *               groups per row). 128 is the common default; a smaller group
 *               follows the weights better at the price of more metadata bits
 *               per weight ("What W4A16 buys ...").
 *   symmetric   0: asymmetric, one b-bit zero point per (row, group);
 *               1: symmetric, zero point fixed at 2^(b-1) (8 or 128), no
 *                  zero points stored.
 *   has_g_idx   0: column k belongs to group k / group_size;
 *               1: GPTQ act order -- a column-to-group map g_idx is given at
 *                  pack time ("The two algorithms, compactly": under act
 *                  order the columns are taken in descending order of their
 *                  activation energy).
 *   N, K        1 <= N <= 2^20, group_size <= K <= 2^20.
 *   has_act_scale 0: none;
 *               1: unfolded AWQ -- the blob carries a per-input-channel
 *                  scale s (fp16 [K], finite, > 0). The weights were
 *                  quantized as fp16(W[n][k] * s[k]) and every product
 *                  divides the activations by s as it loads them:
 *                  y = fp16(x / s) . W_hat^T ("AWQ + GPTQ Quantization, in
 *                  depth", section "The two algorithms, compactly": the
 *                  salient channels' weights are multiplied by s before
 *                  quantizing and the activations divided by it; here the
 *                  division is not folded into the preceding operation).
 *                  Pack with w4a16_pack_awq.
 */
typedef struct {
  int32_t bits;
  int32_t group_size;
  int32_t symmetric;
  int32_t has_g_idx;
  int64_t N;
  int64_t K;
  int32_t has_act_scale;
} w4a16_format;

/*
 * Packed blob (device memory, 256-byte aligned, produced by w4a16_pack).
 * With NR = ceil(N / 128) row blocks, KB = ceil(K / 64) column blocks and
 * G = K / group_size, it holds up to five sub-arrays, each starting on a
 * 256-byte boundary, in this order:
 *   qweight  NR*KB*1024*b bytes: for every (row block, column block) a tile
 *            of 128 rows x 64 columns of b-bit codes (3, 4 or 8 KiB),
 *            arranged so that a warp's 16-byte (3 bits: 16- and 8-byte)
 *            loads yield tensor-core operand fragments.
 *   scales   NR*G*256 bytes: fp16 scales, 128 rows per (row block, group).
 *   zeros    (asymmetric only) NR*G*64 bytes of 4-bit zero points for 3- and
 *            4-bit codes, NR*G*128 bytes of 8-bit ones for 8-bit codes,
 *            arranged like the scales.
 *   perm     K*4 bytes (act order only): packed column -> original column.
 *   act_scale K*2 bytes (has_act_scale only): fp16 s in packed column order.
 * Rows beyond N and columns beyond K are padding. The blob's meaning is fixed
 * by w4a16_dequant; its internal arrangement is private and may change.
 */

/* Bytes the packed blob needs for format f; 0 if f is invalid or unsupported. */
W4A16_API size_t w4a16_packed_bytes(const w4a16_format* f);

/* W4A16_OK if f is valid and supported, else the error w4a16_pack would return. */
W4A16_API w4a16_status w4a16_check_format(const w4a16_format* f);

/* Static, human-readable name of a status code. Never NULL. */
W4A16_API const char* w4a16_status_string(w4a16_status s);

/* cudaError_t of the calling thread's most recent W4A16_ERR_CUDA (0 if none). */
W4A16_API int w4a16_last_cuda_error(void);

/*
 * Round-to-nearest group quantization of fp16 weights (the step before the
 * path: "LLM Quantization: INT8, GPTQ, and AWQ Explained", section "What
 * quantization actually does" -- find each group's range, pick the scale,
 * round to the nearest grid point, clamp). Per (row n, group t), in fp64,
 * with qmax = 2^b - 1:
 *   asymmetric: s = fp16_rne((max - min) / qmax), z = clamp(rint(-min / s), 0, qmax)
 *   symmetric, 3 or 4 bits: s = fp16_rne(2 * max|w| / qmax), z = 2^(b-1)
 *               (4 at 3 bits, 8 at 4 bits)
 *   symmetric, 8 bits: s = fp16_rne(max|w| / 127), z = 128 (the int8 absmax
 *               code of the same section, stored offset by 128), and
 *               q = clamp(rint(w / s), -127, 127) + 128 (codes 1 .. 255)
 *   (s == 0 is replaced by 1.0), otherwise q = clamp(rint(w / s) + z, 0, qmax),
 *   rint = round half to even.
 *   w        fp16 [N][K] row-major, 16-byte aligned.
 *   g_idx    HOST int32 [K] (act order) or NULL; group t's members are the
 *            columns k with g_idx[k] == t, exactly group_size of them.
 *   q        uint8 [N][K] codes 0 .. qmax, original column order.
 *   scales   fp16 [N][G], 2-byte aligned.
 *   zeros    uint8 [N][G]; must be NULL when f->symmetric.
 *   workspace / workspace_bytes: >= w4a16_quantize_workspace_bytes(f)
 *            (K*4 bytes for act order, else 0; may be NULL when 0),
 *            16-byte aligned.
 * With g_idx the call copies a host-built column list to the workspace with
 * cudaMemcpyAsync from pageable memory, so it synchronises with the host.
 */
W4A16_API size_t w4a16_quantize_workspace_bytes(const w4a16_format* f);
W4A16_API w4a16_status w4a16_quantize_rtn(const w4a16_format* f, const uint16_t* w,
                                const int32_t* g_idx, uint8_t* q, uint16_t* scales,
                                uint8_t* zeros, void* workspace, size_t workspace_bytes,
                                w4a16_stream_t stream);

/*
 * w4a16_quantize_rtn for callers that cannot allocate device memory -- for
 * example code inside a framework or plugin that owns every device
 * allocation, or a path that must not allocate at all. The act-order column
 * list that w4a16_quantize_rtn keeps in caller workspace lives here in a fixed
 * 256 KiB array of device memory owned by the library (held by every GPU that
 * loads it until the process exits). The pages have no counterpart; this is a
 * deployment variant only, with the same arguments and results as
 * w4a16_quantize_rtn minus the workspace.
 *   Limit: with act order K <= 65536; larger K returns
 *   W4A16_ERR_BUFFER_TOO_SMALL (without act order there is no limit beyond
 *   the format's).
 *   No cudaMalloc/cudaFree or other allocation, on the device or the host.
 *   The first call with act order on a device looks up the array's device
 *   address (cudaGetSymbolAddress) with that device current; make that first
 *   call before any stream capture. A lookup that fails returns
 *   W4A16_ERR_CUDA and is tried again on the next call.
 *   Every call shares the one array and leaves its column list there. Calls
 *   that may run at the same time on the GPU (different streams, or different
 *   host threads with their own streams) race on it. Calls on one stream do
 *   not, from any number of host threads: a lock is held from the host-side
 *   staging until the call's copy and its kernel are both queued.
 */
W4A16_API w4a16_status w4a16_quantize_rtn_noalloc(const w4a16_format* f, const uint16_t* w,
                                const int32_t* g_idx, uint8_t* q, uint16_t* scales,
                                uint8_t* zeros, w4a16_stream_t stream);

/*
 * Pack canonical codes, scales and zero points into the device blob.
 *   q        uint8 [N][K], codes 0 .. 2^b - 1 (3 and 4 bits: only the low b
 *            bits are used).
 *   scales   fp16 [N][G], 2-byte aligned.
 *   zeros    uint8 [N][G] codes 0 .. 2^b - 1 when asymmetric (3 and 4 bits:
 *            the low 4 bits are stored, so a 3-bit zero point above 7 is
 *            kept as given; it is not checked); NULL when symmetric.
 *   g_idx    HOST int32 [K] when f->has_g_idx, else NULL. Every group
 *            0..G-1 must have exactly group_size members (checked here);
 *            the blob stores the columns sorted by group (stable), so that
 *            each group is contiguous in the packed order.
 *   packed / packed_bytes: 256-byte aligned, >= w4a16_packed_bytes(f).
 * With g_idx the call copies the column order from pageable host memory
 * (cudaMemcpyAsync), so it synchronises with the host.
 */
W4A16_API w4a16_status w4a16_pack(const w4a16_format* f, const uint8_t* q, const uint16_t* scales,
                        const uint8_t* zeros, const int32_t* g_idx, void* packed,
                        size_t packed_bytes, w4a16_stream_t stream);

/*
 * Unfolded AWQ ("The two algorithms, compactly"): the round-to-nearest
 * quantizer applied to fp16_rne(w[n][k] * act_scale[k]) (the fp32 product of
 * two fp16 values is exact, it is rounded once), and the packer that also
 * stores act_scale in the blob. Arguments as for w4a16_quantize_rtn and
 * w4a16_pack, plus
 *   act_scale  fp16 [K] in original column order, 2-byte aligned, every
 *              value finite and > 0 (not checked on the device: a zero or
 *              negative scale gives undefined outputs).
 * f->has_act_scale must be 1. w4a16_pack and w4a16_quantize_rtn reject a
 * format with has_act_scale = 1 (W4A16_ERR_INVALID_ARG), so a blob cannot
 * lose its scale by accident.
 */
W4A16_API w4a16_status w4a16_quantize_rtn_awq(const w4a16_format* f, const uint16_t* w,
                                const uint16_t* act_scale, const int32_t* g_idx, uint8_t* q,
                                uint16_t* scales, uint8_t* zeros, void* workspace,
                                size_t workspace_bytes, w4a16_stream_t stream);
W4A16_API w4a16_status w4a16_pack_awq(const w4a16_format* f, const uint8_t* q, const uint16_t* scales,
                        const uint8_t* zeros, const int32_t* g_idx, const uint16_t* act_scale,
                        void* packed, size_t packed_bytes, w4a16_stream_t stream);

/*
 * GPTQ ("AWQ + GPTQ Quantization, in depth", section "The two algorithms,
 * compactly"): quantize the layer one input column at a time; each column's
 * rounding error is compensated on the remaining (later) columns, with weights
 * taken from the inverse of H = 2 X X^T of the calibration activations. On the device, in
 * fp64: H, H += damp * mean(diag H) * I (a channel whose activations are all
 * zero gets diag 1 first), the upper Cholesky factor U of H^-1, then per
 * column j (in order, or -- f->has_g_idx -- by descending diag H, ties to the
 * lower column) q_j = the group's grid point of the current w_j,
 * W[:, j+1:] -= (w_j - q_j) / U[j, j] * U[j, j+1:]. A group's scale and zero
 * point are set when its first column is reached, from the current weights of
 * its columns, with the round-to-nearest rules of w4a16_quantize_rtn.
 *   w        fp16 [N][K], 2-byte aligned (read only).
 *   x        fp16 [T][K] calibration activations, 1 <= T <= 2^24.
 *   damp     >= 0 (0.01 on the page).
 *   q, scales, zeros   as from w4a16_quantize_rtn (codes in original column
 *            order; group t = the t-th run of group_size columns in
 *            processing order).
 *   g_idx    device int32 [K] (written) when f->has_g_idx -- the act-order
 *            column-to-group map to give w4a16_pack (copied to the host) --,
 *            else NULL.
 *   workspace: >= w4a16_gptq_workspace_bytes(f) (2 K^2 + N K doubles and a
 *            little more), 256-byte aligned.
 * Asynchronous on `stream`. Formats with an act scale: W4A16_ERR_UNSUPPORTED.
 */
W4A16_API size_t w4a16_gptq_workspace_bytes(const w4a16_format* f);
W4A16_API w4a16_status w4a16_gptq(const w4a16_format* f, const uint16_t* w, const uint16_t* x, int64_t T,
                        double damp, uint8_t* q, uint16_t* scales, uint8_t* zeros, int32_t* g_idx,
                        void* workspace, size_t workspace_bytes, w4a16_stream_t stream);

/*
 * Expand the blob to fp16 weights: w_out[n][k] = fp16_rne((q - z) * s), in
 * the original column order; bit-exact ("The Math of Quantization":
 * x_approx = (q - Z) * S, rounded once to fp16).
 *   w_out    fp16 [N][K] row-major, 16-byte aligned.
 */
W4A16_API w4a16_status w4a16_dequant(const w4a16_format* f, const void* packed, size_t packed_bytes,
                           uint16_t* w_out, w4a16_stream_t stream);

/*
 * Decode-sized product y = x . W_hat^T for 1 <= M <= 16 tokens: every packed
 * weight is read from HBM once, expanded in registers and multiplied on the
 * tensor cores with fp32 accumulation ("What W4A16 buys ...": one token at
 * batch one reads every weight once, about two flops per weight, so decode
 * is bandwidth-bound).
 *   x        fp16 [M][K] row-major, 16-byte aligned.
 *   y        fp16 [M][N] row-major, 16-byte aligned; must not overlap x.
 * Error per element is within 2e-3 * sum_k |x[m][k] * W_hat[n][k]| + 1e-3 of
 * the exact product with the dequantized weights (with an act scale: x
 * replaced by fp16_rne(x / s), rounded once, in both places). Under act
 * order, with an act scale, or when K is not a multiple of 64 a thread block
 * gathers its slice of x into shared memory (dividing by s there), which
 * bounds M * K / ksplit; a shape beyond that bound returns
 * W4A16_ERR_UNSUPPORTED.
 */
W4A16_API w4a16_status w4a16_gemv(const w4a16_format* f, const void* packed, size_t packed_bytes,
                        const uint16_t* x, uint16_t* y, int64_t M, w4a16_stream_t stream);

/*
 * Grouped decode product: n (1..4) layers that read the same activations x
 * (the q, k and v projections of a decoder layer, or gate and up) in one
 * launch; y[m] = x . W_hat_m^T, each as w4a16_gemv (same bound). The layers
 * share K, bits, group_size and symmetric (else W4A16_ERR_INVALID_ARG) and
 * have neither act order nor an act scale (else W4A16_ERR_UNSUPPORTED); N
 * may differ. formats, packed, packed_bytes and y are HOST arrays of n
 * entries; x, packed[m] and y[m] are device pointers aligned as for
 * w4a16_gemv. flags: as w4a16_gemv_ex (W4A16_GEMV_STAGE_ACTIVATIONS
 * excepted). The launch shape is chosen for the group as a whole.
 */
W4A16_API w4a16_status w4a16_gemv_grouped(const w4a16_format* formats, const void* const* packed,
                                const size_t* packed_bytes, int32_t n, const uint16_t* x,
                                uint16_t* const* y, int64_t M, uint32_t flags, w4a16_stream_t stream);

/*
 * Chained decode products: one persistent launch computes y_i = x_i . W_hat_i^T
 * for a list of layers (1 <= M <= 16 tokens each), e.g. every linear of a
 * decoder stack for one token step. Each layer is the decode product of
 * w4a16_gemv, with the same error bound; what the chain adds is the launch
 * ("What W4A16 buys ...": decode is bandwidth-bound, so time between layers
 * -- launch ramp-up, drain, dependency waits -- is lost bandwidth):
 *   - one thread block per SM; every layer is cut into row groups of 32 rows
 *     and each block owns a contiguous share of them (full K), the shares
 *     rotated from layer to layer so that every SM streams the same bytes;
 *   - a TMA producer per block streams the block's packed weights, scales and
 *     zero points layer after layer into a shared-memory ring, without ever
 *     waiting for a dependency (weights do not depend on earlier layers);
 *   - the block's compute warps read a layer's activations only once every
 *     layer it depends on has been completed by every block (device-side
 *     completion counters); a finishing warp adds the warps' partial sums in
 *     a fixed order and writes y.
 * Results are deterministic for a given device.
 *
 *   w4a16_chain_layer: packed / packed_bytes (one blob per layer), x
 *            (fp16 [M][K], 16-byte aligned) and y (fp16 [M][N], 16-byte
 *            aligned), and the inclusive range [wait_lo, wait_hi] of earlier
 *            layers (indices < this layer's) whose outputs this layer reads:
 *            its activations are read only after every one of those layers
 *            has written all of its y. wait_lo > wait_hi: no dependency (x is
 *            ready before the launch). Any other overlap between a layer's y
 *            and another's x or y is the caller's to avoid.
 *   formats  one w4a16_format per layer. All layers share bits, group_size
 *            and symmetric; none has act order or an act scale, and K is a
 *            multiple of 64 (else W4A16_ERR_UNSUPPORTED).
 *   workspace: >= w4a16_chain_workspace_bytes(formats, n_layers, M) bytes
 *            (counters, the table of layer slices and the TMA tensor maps of
 *            every blob), 256-byte aligned, device memory the chain owns from
 *            prepare until the last run; the size is 0 for an invalid or
 *            unsupported list. It does not depend on the device.
 *
 * w4a16_chain_prepare validates everything on the host, then -- for the
 * current device -- cuts layers too large for one pass into slices, encodes
 * the tensor maps and writes the table into the workspace with synchronous
 * host-to-device copies, and fills *info (host memory, caller-owned). The
 * blobs must not move afterwards (the tensor maps hold their addresses).
 * w4a16_chain_run then resets the counters and launches the chain on `stream`
 * (both asynchronous; may be captured in a CUDA graph), on a device with the
 * SM count it was prepared for (else W4A16_ERR_INVALID_ARG). Every wait
 * inside the launch is bounded (1 s, see w4a16_set_wait_limit_ns); a wait
 * that gives up stops every block,
 * leaves the outputs undefined and is counted (w4a16_pipeline_timeouts). The
 * launch needs one resident thread block per SM (cooperative launch); it
 * fails with W4A16_ERR_CUDA rather than wait if the device cannot host them.
 */
typedef struct {
  const void* packed;
  size_t packed_bytes;
  const uint16_t* x;
  uint16_t* y;
  int32_t wait_lo;
  int32_t wait_hi;
} w4a16_chain_layer;

typedef struct {
  int32_t n_layers;
  int32_t bits;
  int32_t group_size;
  int32_t symmetric;
  int64_t M;
  int64_t n_slices;  /* entries of the slice table (>= n_layers) */
  int32_t blocks;    /* thread blocks (SMs of the device) the table was planned for */
  int32_t flags;     /* set by prepare for run: activation buffers in shared memory (0 or 2) */
  int32_t reserved_x;/* set by prepare for run: bytes of the area the two buffers share */
  int32_t reserved;
} w4a16_chain_info;

W4A16_API size_t w4a16_chain_workspace_bytes(const w4a16_format* formats, int32_t n_layers, int64_t M);
W4A16_API w4a16_status w4a16_chain_prepare(const w4a16_format* formats, const w4a16_chain_layer* layers,
                                 int32_t n_layers, int64_t M, void* workspace, size_t workspace_bytes,
                                 w4a16_chain_info* info);
W4A16_API w4a16_status w4a16_chain_run(const w4a16_chain_info* info, void* workspace,
                             w4a16_stream_t stream);

/*
 * Prefill-sized product y = x . W_hat^T for M >= 1 tokens on the tcgen05
 * tensor cores ("AWQ + GPTQ Quantization, in depth", section "What W4A16 buys
 * and why decoding gets faster": the 4-bit weights are expanded to 16 bits
 * before the multiply; with many tokens the product is compute-bound). The
 * weights are dequantized -- w_hat = fp16((q - z) * s), the same values as
 * w4a16_dequant -- straight into tensor memory, where they are the MMA's A
 * operand; the activations are streamed by TMA; fp32 accumulators live in
 * tensor memory. Same arguments and error bound as w4a16_gemv, plus
 *   workspace / workspace_bytes: >= w4a16_gemm_workspace_bytes(f, M)
 *            (the activations reordered to the packed column order and
 *            divided by the act scale, when the format has act order or an
 *            act scale: M*K*2 bytes; else 0, may be NULL),
 *            16-byte aligned, overlapping neither x nor y.
 * 1 <= M <= 2^20. Needs a Blackwell GPU (compute capability 10.x); returns
 * W4A16_ERR_UNSUPPORTED on older devices.
 * Every pipeline wait inside the kernel is bounded (1 s, see
 * w4a16_set_wait_limit_ns); a wait that gives up leaves y unwritten for its
 * tile and is counted on the device, see w4a16_pipeline_timeouts().
 */
W4A16_API size_t w4a16_gemm_workspace_bytes(const w4a16_format* f, int64_t M);
W4A16_API w4a16_status w4a16_gemm(const w4a16_format* f, const void* packed, size_t packed_bytes,
                        const uint16_t* x, uint16_t* y, int64_t M, void* workspace,
                        size_t workspace_bytes, w4a16_stream_t stream);

/*
 * w4a16_gemm with the launch shape chosen by the caller:
 *   tile    0 = default, 1 = 128 weight rows x 256 tokens per thread block,
 *           2 = 256 x 128, 3 = 128 x 256 with twice the dequantization warps
 *           of 1, 4 = 128 x 256 with half of them, 5 = 128 x 128 and
 *           6 = 128 x 64 (two thread blocks per SM).
 *   ksplit  thread blocks of a cluster that split K (1, 2, 4, 8 or 16; their
 *           fp32 partial sums are added in rank order through distributed
 *           shared memory); 0 = default (1 when `tile` is given).
 * By default up to 64 tokens use tile 6, up to 128 tile 5 and more tokens
 * tile 1, with K split so that the grid covers the SMs (at least 8 steps of
 * 64 columns per thread block). Results match w4a16_gemm's within the
 * error bound (the summation order depends on ksplit).
 */
W4A16_API w4a16_status w4a16_gemm_ex(const w4a16_format* f, const void* packed, size_t packed_bytes,
                           const uint16_t* x, uint16_t* y, int64_t M, void* workspace,
                           size_t workspace_bytes, int32_t tile, int32_t ksplit,
                           w4a16_stream_t stream);

/*
 * Number of bounded pipeline waits on the current device that gave up since
 * the previous call (each one means a tile of some w4a16_gemm output, or the
 * later outputs of a chained launch, were not written); the count is reset.
 * Synchronous: waits for the device's pending work to finish. Not expected to
 * be nonzero in correct operation. Whenever it is nonzero, the outputs of the
 * launches it covers are undefined, and so is any timing taken of them.
 */
W4A16_API w4a16_status w4a16_pipeline_timeouts(uint32_t* count);

/*
 * Limit, in nanoseconds, of every bounded pipeline wait inside the kernels
 * (w4a16_gemm, w4a16_chain_run) launched after this call; 0 restores the
 * default, 1 s. Returns the previous limit. Process-wide. A launch captured in
 * a CUDA graph keeps the limit in force when it was captured. Meant for tests
 * of the timeout path: a limit shorter than the work the waits cover makes
 * them give up (counted by w4a16_pipeline_timeouts, outputs undefined) and the
 * launch return; waits that only let copies already issued land before a
 * thread block exits keep their own 1 s.
 */
W4A16_API uint64_t w4a16_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook: the next call (from any thread) that would launch device work
 * launches nothing and returns W4A16_ERR_CUDA, with w4a16_last_cuda_error()
 * == error in the calling thread. One-shot; 0 clears a pending error. Lets a
 * caller's handling of a failed launch be tested without a device fault.
 */
W4A16_API void w4a16_debug_fail_next_launch(int error);

/*
 * Debug flavor of the library (libw4a16_debug.so, built with
 * -DW4A16_DEBUG_CHECKS): the decode stream checks the indices of its code,
 * scale and zero-point copies, of the staged activations and group sums, of
 * the slot units and of the partial sums it reads and writes; a failed check
 * skips the access and records its code (the first one wins; 0x1xx producer,
 * 0x2xx staging, 0x3xx consumer warps, 0x4xx layer shares). Synchronizes the
 * device, then stores the recorded code (0: none) in *word and resets it.
 * W4A16_ERR_UNSUPPORTED (and *word = 0) in the release library.
 */
W4A16_API w4a16_status w4a16_debug_check_word(uint32_t* word);

/*
 * w4a16_gemv with options.
 *   shape    16-row tiles per thread block, 2, 4 or 8; 0 = default.
 *   ksplit   thread blocks per cluster splitting K: 1, 2, 4, 8 or 16;
 *            0 = default.
 *   flags    0 or an OR of
 *            W4A16_GEMV_WEIGHTS_READY: no kernel still in flight on the
 *              stream writes `packed` (true once the weights were packed
 *              before the preceding kernel started, as in a decode loop);
 *              the GEMV then starts streaming weights before the previous
 *              kernel finishes. `x` is always read after it.
 *            W4A16_GEMV_INPUTS_READY: stronger than WEIGHTS_READY: no
 *              kernel still in flight on the stream writes `packed` or `x`,
 *              or reads or writes `y` (for example k and v after q, which
 *              read the same activations). The GEMV then does not wait for
 *              the previous kernel at all and may run alongside it. A later
 *              kernel that waits for this GEMV through programmatic
 *              dependent launch no longer waits, through it, for the kernels
 *              before it; work that depends on those must follow an
 *              ordinary stream dependency.
 *            W4A16_GEMV_REGISTER_RING: the kernel that loads the next weight
 *              units straight into a ring of registers.
 *            W4A16_GEMV_ASYNC_COPY: the kernel in which every thread lands
 *              its next units (codes, scales, zero points) with asynchronous
 *              copies (cp.async) in a ring of shared-memory slots instead of
 *              registers (more bytes in flight per SM).
 *            W4A16_GEMV_STAGE_ACTIVATIONS: copy each thread block's
 *              activations to shared memory before the weight stream.
 * Without REGISTER_RING or ASYNC_COPY, layers of at least 64 row blocks of
 * 128 (N > 8064) use the asynchronous-copy kernel and smaller ones the
 * register ring (measured on B300); w4a16_gemv always takes that default.
 * The GEMV kernels are launched with programmatic dependent launch, so a GEMV
 * may start while the previous kernel on the stream is still running; by
 * default it reads nothing from global memory before that kernel is done.
 * Results equal w4a16_gemv's up to summation order.
 */
#define W4A16_GEMV_WEIGHTS_READY 1u
#define W4A16_GEMV_REGISTER_RING 2u
#define W4A16_GEMV_STAGE_ACTIVATIONS 4u
#define W4A16_GEMV_ASYNC_COPY 8u
#define W4A16_GEMV_INPUTS_READY 16u
W4A16_API w4a16_status w4a16_gemv_ex(const w4a16_format* f, const void* packed, size_t packed_bytes,
                           const uint16_t* x, uint16_t* y, int64_t M, int32_t shape,
                           int32_t ksplit, uint32_t flags, w4a16_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
