/*
 * bit1.h -- C ABI of the true 1-bit linear-layer library for NVIDIA B300
 * (sm_103a).
 *
 * The weight format (web page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진
 * 및 삼진 저비트 LLM (feat. PrismML)", section "이진(Binary) 가중치 형식"):
 * every weight is w = s_g * b with b in {-1, +1}; each run of 128 consecutive
 * input-dimension weights of a row shares one FP16 scale s_g, so a weight
 * costs 1 + 16/128 = 1.125 bits.  The same page ("저장 공간과 실제 배포 크기")
 * deploys binary weights in their native 1-bit layout, and its kernel section
 * ("하이브리드 어텐션을 위한 저비트 커널") decodes the sign codes and applies
 * the group scale inside the fused product, never rebuilding a dense FP16
 * matrix, with high-precision accumulation.  The row-wise XOR patch follows
 * "LocalLLaMA, true 1-bit LLM용 XOR patch 방식 \"Bankai\" 실험에 주목",
 * section "LocalLLaMA가 본 핵심 포인트".
 *
 * Layout (the pages do not fix one; this library's reading):
 *   bits   : uint8 [N][K/8], row-major; bit k of row n is
 *            (bits[n*K/8 + k/8] >> (k%8)) & 1, i.e. least significant bit
 *            first; bit 1 means +1, bit 0 means -1.  Seen as little-endian
 *            32-bit words, bit k of a row is bit (k%32) of word k/32, and the
 *            16 bytes at offset 16*g of a row hold group g exactly.
 *   scales : IEEE binary16 bit patterns [N][K/128], row-major.
 *   x      : bfloat16 [B][K], row-major (activations).
 *   y      : [B][N] row-major, fp32 or bf16 (round to nearest even).
 *   K must be a positive multiple of 128.
 *
 * Ownership and execution: the caller owns every buffer.  Device pointers
 * must point to device memory of the current device and be 16-byte aligned.
 * No entry point allocates device memory; bit1_gemv takes an optional
 * caller-owned workspace.  Every call is asynchronous on `stream` (NULL means
 * the legacy default stream) and validates its arguments on the host before
 * launching anything: a call that returns an error has launched nothing and
 * modified nothing.  Errors of kernels that have already been launched
 * surface at the caller's next synchronisation, as usual in CUDA.
 */
#ifndef BIT1_H
#define BIT1_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *bit1_stream_t;

typedef enum bit1_status {
    BIT1_OK = 0,
    BIT1_EINVAL = 1, /* null or misaligned pointer, unknown dtype/variant, bad count */
    BIT1_ESHAPE = 2, /* B, N < 1; K not a positive multiple of 128; shape beyond a variant's limits */
    BIT1_ERANGE = 3, /* patch row outside [0, N); packed scale not finite; ternary code not -1/0/+1 */
    BIT1_ECUDA = 4,  /* a CUDA runtime call or kernel launch failed */
    BIT1_ENAN = 5    /* NaN among the weights given to bit1_pack */
} bit1_status;

enum bit1_dtype {
    BIT1_F32 = 0,
    BIT1_BF16 = 1,
    BIT1_F16 = 2
};

/* Kernel selection for bit1_gemv_ex.  AUTO picks by shape (the same choice
 * bit1_gemv makes); the others force one kernel and return BIT1_ESHAPE if
 * that kernel cannot take the shape.  AUTO, from per-call times measured on
 * one B300: the tensor cores when the workspace allows them and they are the
 * faster (B >= 16; B >= 8; B >= 4 for N <= 8192; B >= 5 for N*K >= 64M;
 * any B >= 2 where the 6-bit tables cannot split K), else at batch 1 the
 * nibble-table kernel below 65536 rows, else the 6-bit tables (the MMA
 * variant from B = 12 at K <= 4096), else the grouped kernel with the one
 * problem (MMA from B = 3, STREAM below), else one warp per row. */
enum bit1_gemv_variant {
    BIT1_GEMV_AUTO = 0,
    BIT1_GEMV_SIMPLE = 1,  /* any shape; one warp per row (reference-quality) */
    BIT1_GEMV_LUT = 2,     /* batch 1..8: CUDA-core table-lookup kernel */
    BIT1_GEMV_SPLITK = 3,  /* the split-K kernel by name: the same kernel as
                              BIT1_GEMV_LUT6, whose K split over a cluster
                              (fixed-order DSMEM reduction, no workspace) and,
                              for short N, over the warps of a CTA, is this
                              library's split-K variant */
    BIT1_GEMV_TC = 4,      /* batch >= 16: tcgen05 tensor-core kernel */
    BIT1_GEMV_LUT6 = 5,    /* K a multiple of 1024: one row per lane, 6-bit fp16
                              tables per batch row, TMA-staged weights, K split
                              over a thread-block cluster; up to 8 batch rows
                              per launch (larger batches: several launches) */
    BIT1_GEMV_STREAM = 6,  /* K a multiple of 1024: the grouped kernel below
                              with the one problem (one CTA per SM streaming a
                              contiguous row range, full-K tables, no clusters;
                              no workspace); up to 6 batch rows per launch
                              (larger batches: ceil(B / 6) launches of
                              balanced row counts) */
    BIT1_GEMV_MMA = 7      /* K a multiple of 1024: the grouped kernel with the
                              one problem on register-sourced tensor-core MMAs
                              (bit1_group_plan_mma's engine; no workspace); up
                              to 16 batch rows per launch (larger batches:
                              ceil(B / 16) launches of balanced row counts) */
};

/* bit1_gemv_ex flags. */
#define BIT1_FLAG_PDL 1u   /* launch with programmatic dependent launch: the
                              kernel prefetches its weights before waiting for
                              the preceding kernel in the stream */
#define BIT1_FLAG_SWIGLU 2u /* the matrix is a SwiGLU MLP's gate and up
                              projections with interleaved rows (row 2n gate,
                              row 2n+1 up of hidden unit n; N even, else
                              BIT1_ESHAPE) and y receives h = silu(g) * u,
                              [B][N/2], as BIT1_EPI_SWIGLU below.  Every
                              variant but BIT1_GEMV_SIMPLE (BIT1_ESHAPE) takes
                              it within its own shape limits; AUTO picks LUT
                              (K <= 13312, else STREAM) at batch 1 and its
                              usual choice otherwise.
                              bit1_gemv_ternary applies it in its combine
                              step instead (any batch, any variant). */

/* ------------------------------------------------------------------------
 * bit1_pack -- floating-point weights -> packed sign bits + fp16 scales.
 * Follows the binary weight format above.  The pages do not say how a scale
 * is chosen from real weights; this library's reading: bit = !(w < 0) (so
 * +0 and -0 give +1), s_g = fp16 round-to-nearest-even of mean(|w|) over
 * the group, the 128 magnitudes summed in fp64 in ascending k order
 * (the least-squares scale for w ~ s*sign(w)).
 *   w       : device, [N][K] of w_dtype (BIT1_F32, BIT1_BF16 or BIT1_F16)
 *   bits    : device, N*K/8 bytes (written)
 *   scales  : device, N*(K/128) fp16 patterns (written)
 *   d_flags : device pointer to one uint32, or NULL.  The call zeroes it on
 *             `stream`; the kernel sets bit 0 if any weight is NaN and bit 1
 *             if any scale is not finite (|mean| beyond fp16 range).  After
 *             synchronising, bit1_pack_flags_status() maps it to a status.
 * Returns BIT1_ESHAPE / BIT1_EINVAL on bad arguments (nothing launched),
 * BIT1_ECUDA on launch failure, else BIT1_OK.
 */
bit1_status bit1_pack(const void *w, int w_dtype, int64_t N, int64_t K,
                      uint8_t *bits, uint16_t *scales, uint32_t *d_flags,
                      bit1_stream_t stream);

/* BIT1_ENAN if bit 0 is set, else BIT1_ERANGE if bit 1 (bit1_pack), bit 2
 * (a ternary code out of range) or bit 3 (a packed ternary byte out of
 * range) is set, else BIT1_OK. */
bit1_status bit1_pack_flags_status(uint32_t flags);

/* ------------------------------------------------------------------------
 * bit1_gemv -- y[b][n] = sum_g s[n][g] * sum_{k in group g} (bit(n,k) ? +x[b][k]
 *                                                             : -x[b][k])
 * The product of the binary weight format above with bf16 activations, the
 * sign decoded and the group scale applied inside the kernel, fp32
 * accumulation (kernel section of the Bonsai 27B page).  Result within
 * 1e-3 * sum_k |s*x_k| + 1e-6 of the exact value (plus the bf16 output
 * rounding for y_dtype = BIT1_BF16).
 *   bits, scales : device, layout above
 *   x            : device, bf16 [B][K]
 *   y            : device, [B][N] of y_dtype (BIT1_F32 or BIT1_BF16), written
 *   workspace    : device scratch of ws_bytes bytes, or NULL/0.  Some shapes
 *                  run faster with bit1_gemv_workspace_bytes(B, N, K) bytes;
 *                  with less, a kernel without scratch is chosen.  Its
 *                  contents on entry do not matter.
 * B >= 1, N >= 1, K a positive multiple of 128.  The inputs must not overlap
 * y or the workspace.
 */
bit1_status bit1_gemv(const uint8_t *bits, const uint16_t *scales,
                      const uint16_t *x, int64_t B, int64_t N, int64_t K,
                      void *y, int y_dtype, void *workspace, size_t ws_bytes,
                      bit1_stream_t stream);

/* bit1_gemv with an explicit kernel choice (enum bit1_gemv_variant) and
 * flags (BIT1_FLAG_*). */
bit1_status bit1_gemv_ex(const uint8_t *bits, const uint16_t *scales,
                         const uint16_t *x, int64_t B, int64_t N, int64_t K,
                         void *y, int y_dtype, void *workspace, size_t ws_bytes,
                         int variant, unsigned flags, bit1_stream_t stream);

/* Scratch bytes that let bit1_gemv use its fastest kernel for this shape
 * (0 when no kernel needs scratch).  On the tensor cores (where AUTO takes
 * them, see enum bit1_gemv_variant) this is
 * the fp16 copy of every batch row's activations plus one float per row,
 * so a batch beyond 64 rows runs as one launch pair; any workspace of at
 * least one 64-row chunk's share (16 * ceil(min(B, 64) / 16) * K * 2 bytes
 * rounded up to 256, plus 256) still selects the tensor cores and runs one
 * launch pair per 64-row chunk. */
size_t bit1_gemv_workspace_bytes(int64_t B, int64_t N, int64_t K);

/* The variant bit1_gemv picks for this shape and workspace size, and the
 * number of kernel launches one call makes with bit1_gemv_workspace_bytes of
 * scratch (0 on bad arguments). */
int bit1_gemv_pick(int64_t B, int64_t N, int64_t K, size_t ws_bytes);
int bit1_gemv_launches(int64_t B, int64_t N, int64_t K, int variant);

/* ------------------------------------------------------------------------
 * Grouped GEMV: many independent batch-1 products in one persistent launch.
 * A decode step reads every weight once, and at batch 1 launch and
 * synchronisation latency, not bandwidth, dominates per-matrix launches (web
 * page "Bonsai 27B: 노트북과 폰에서 실행되는 27B급 이진 및 삼진 저비트 LLM",
 * section "하이브리드 어텐션을 위한 저비트 커널").  Each problem is one
 * bit1_gemv with B = 1; the problems must not depend on each other (no y is
 * another problem's x).  K must be a multiple of 1024; y_dtype BIT1_F32 or
 * BIT1_BF16; all pointers device pointers, 16-byte aligned.
 *
 * Use: bit1_group_plan() encodes the problems (TMA descriptors and a
 * cost-balanced split of all rows over the SMs) into a caller-owned HOST
 * buffer of bit1_group_plan_bytes(count) bytes (128-byte aligned).  The caller
 * copies it, unchanged, into a DEVICE buffer of the same size (128-byte
 * aligned) and then calls bit1_gemv_group(device_plan, host_plan, ...) as
 * often as it likes (the plan embeds the problems' pointers and shapes: it is
 * valid while those buffers are).  Results are bit-identical to running the
 * problems one by one with BIT1_GEMV_STREAM.
 */
typedef struct bit1_gemv_problem {
    const uint8_t *bits;     /* [N][K/8] sign bits */
    const uint16_t *scales;  /* [N][K/128] fp16 scales */
    const uint16_t *x;       /* [K] bf16 activations */
    void *y;                 /* [N] output of y_dtype ([N/2] with BIT1_EPI_SWIGLU) */
    int64_t N, K;
    int y_dtype;
    int epilogue;            /* BIT1_EPI_NONE (0) or BIT1_EPI_SWIGLU; other values: BIT1_ESHAPE */
} bit1_gemv_problem;

/* Epilogue of a grouped problem.  BIT1_EPI_SWIGLU: the problem is the gate and
 * up projections of a SwiGLU MLP (the Bonsai 27B page, section "Bonsai 27B의
 * 표현 방식": the base model keeps its SwiGLU MLP, and the MLP projections are
 * binary like the rest) stored as ONE matrix with interleaved rows -- row 2n
 * the gate, row 2n+1 the up projection of hidden unit n; N (the interleaved
 * row count) must be even, else BIT1_ESHAPE.  y then receives
 *     h[b][n] = silu(g) * u,  silu(g) = g / (1 + exp(-g)),
 * [B][N/2] of y_dtype, computed in fp32 from the fp32 gate and up results
 * before the one output rounding; the gate and up values are not written.
 * Error: the GEMV error of g and u carried through h (|silu'| <= 1.1) plus a
 * few fp32 ulps of h. */
#define BIT1_EPI_NONE   0
#define BIT1_EPI_SWIGLU 1

size_t bit1_group_plan_bytes(int count);
bit1_status bit1_group_plan(const bit1_gemv_problem *problems, int count,
                            void *host_plan, size_t plan_bytes);

/* The same with B batch rows per problem (1 <= B <= 6, else BIT1_ESHAPE):
 * every problem's x is bf16 [B][K] and its y is [B][N] (row-major, y_dtype),
 * all problems sharing B.  This is the batched verify pass of a speculative
 * drafter (the Bonsai 27B page, section "DSpark: 추측 디코딩으로 한 번 더
 * 가속": the target model checks the k drafted tokens in one multi-row pass).
 * The whole weight set runs once for all B rows: the sign bits of a group are
 * read once and looked up in every row's tables.  Same plan buffer size and
 * the same bit1_gemv_group call. */
bit1_status bit1_group_plan_batched(const bit1_gemv_problem *problems, int count,
                                    int B, void *host_plan, size_t plan_bytes);
/* The same with an explicit sign-bit layout shared by every problem of the
 * plan: BIT1_LAYOUT_CANONICAL (the layout above; bit1_group_plan and
 * bit1_group_plan_batched) or BIT1_LAYOUT_G128X (bits converted with
 * bit1_repack_g128x, below).  1 <= B <= 6.  BIT1_EINVAL for another layout
 * value; otherwise as bit1_group_plan_batched.  Results do not depend on the
 * layout: each field of six inputs is looked up in the same table either
 * way, only its position in the 16 bytes of the group differs. */
#define BIT1_LAYOUT_CANONICAL 0
#define BIT1_LAYOUT_G128X     1
bit1_status bit1_group_plan_ex(const bit1_gemv_problem *problems, int count, int B,
                               int layout, void *host_plan, size_t plan_bytes);

/* The same batched grouped product (canonical layout, 1 <= B <= 16, else
 * BIT1_ESHAPE) on register-sourced tensor-core MMAs (mma.sync m16n8k16,
 * fp16 operands, fp32 accumulation): weights become +-s in fp16 registers,
 * each problem's activations are converted per K chunk of 2048 (B <= 8) or
 * 1024 inputs (B > 8) to fp16 with an exact per-row power-of-two prescale,
 * and the batch rows are the MMA's columns, so the work per weight does not
 * grow with B.  Same plan buffer size and the same bit1_gemv_group call;
 * results agree with the table engine within the GEMV tolerance (different
 * summation order) and are deterministic run to run. */
bit1_status bit1_group_plan_mma(const bit1_gemv_problem *problems, int count, int B,
                                void *host_plan, size_t plan_bytes);

/* Runs a plan made by any bit1_group_plan* call above or below (the plan
 * records which kernel it is for).  flags: BIT1_FLAG_PDL or 0. */
bit1_status bit1_gemv_group(const void *device_plan, const void *host_plan,
                            unsigned flags, bit1_stream_t stream);

/* Grouped products on the tensor cores: the same problems (bit1_gemv_problem,
 * same rules: K a multiple of 1024, 16-byte aligned device pointers, row-major
 * x [B][K] bf16 and y [B][N] or [B][N/2] with BIT1_EPI_SWIGLU) at a batch of
 * 1 <= B <= 64 rows shared by every problem (else BIT1_ESHAPE), for the
 * multi-row verify pass of speculative decoding (the Bonsai 27B page,
 * section "DSpark: 추측 디코딩으로 한 번 더 가속") and batched decode.  The
 * arithmetic is bit1_gemv's BIT1_GEMV_TC path: weights +-s in fp16, the
 * activations as fp16 with an exact per-row power-of-two prescale, fp32
 * accumulation on the tensor cores; results equal BIT1_GEMV_TC's within the
 * same tolerance (the summation order inside an MMA is the hardware's).
 *
 * Use: a caller-owned DEVICE workspace of bit1_group_tc_workspace_bytes()
 * bytes (256-byte aligned; it receives the activations' fp16 copies on every
 * run) and a HOST plan buffer of bit1_group_tc_plan_bytes(count) bytes
 * (128-byte aligned); bit1_group_plan_tc() fills the plan, which the caller
 * copies unchanged into a device buffer of the same size and runs with
 * bit1_gemv_group (two launches: the activation prep, then one persistent
 * kernel over all problems).  The plan embeds the problems' pointers and the
 * workspace's: valid while those buffers are; runs of one plan must not
 * overlap in time (they share the workspace).  Errors: BIT1_EINVAL for null
 * or misaligned buffers or a workspace or plan buffer that is too small;
 * BIT1_ESHAPE for a problem outside the rules or B outside [1, 64];
 * BIT1_ECUDA if a tensor map cannot be encoded.  bit1_group_tc_workspace_bytes
 * returns 0 on invalid arguments. */
size_t bit1_group_tc_plan_bytes(int count);
size_t bit1_group_tc_workspace_bytes(const bit1_gemv_problem *problems, int count, int B);
bit1_status bit1_group_plan_tc(const bit1_gemv_problem *problems, int count, int B,
                               void *workspace, size_t ws_bytes, void *host_plan,
                               size_t plan_bytes);

/* ------------------------------------------------------------------------
 * bit1_repack_g128x / bit1_unpack_g128x -- convert packed sign bits between
 * the canonical layout and the g128x layout, a fixed permutation of the 128
 * bits of every group (the pages fix no bit layout beyond "packed 1-bit";
 * this one is this library's, chosen for the cost of reading it):
 *   input k of a group (0 <= k < 128), canonical bit k, is stored at
 *     k <  72:  bit 8*(k/6) + 1 + k%6                 (bits 1-6 of bytes 0..11)
 *     k <  96:  j = (k-72)/6, i = (k-72)%6, in word i/2 (bytes 4*(i/2)..),
 *               bit 7 of byte j if i is even, else bit 0 of byte (j+1)%4
 *     k >= 96:  bit k                                  (word 3 unchanged)
 * (bit b of the group is bit b%8 of byte b/8).  The grouped kernel then forms
 * each lookup index of bytes 0..11 with one byte permute instead of a shift
 * and a mask.  Rows keep their own bits, so bit1_xor_patch flips the same
 * rows in either layout and applying it commutes with the conversion; the
 * scales are not touched.  Only plans built with BIT1_LAYOUT_G128X read the
 * g128x layout; every other call takes the canonical one.
 *   bits : device [N][K/8] in the source layout; out: device [N][K/8] (may
 *          be bits itself: converted in place).  16-byte aligned.
 * BIT1_ESHAPE for K not a multiple of 128 (or N, K < 1); BIT1_EINVAL for a
 * null or misaligned pointer.  Asynchronous on `stream`.  Allocates nothing.
 */
bit1_status bit1_repack_g128x(const uint8_t *bits, int64_t N, int64_t K, uint8_t *out,
                              bit1_stream_t stream);
bit1_status bit1_unpack_g128x(const uint8_t *bits, int64_t N, int64_t K, uint8_t *out,
                              bit1_stream_t stream);

/* ------------------------------------------------------------------------
 * bit1_xor_patch -- the Bankai row-wise sign-flip patch, in place.
 * Every listed row has all of its K sign bits inverted (bytes ^= 0xFF);
 * scales are untouched.  Applying the same list again removes the patch.
 * A row listed twice is flipped twice (no change).
 *   bits   : device, [N][K/8] (modified in place)
 *   rows   : HOST array of n_rows row indices (the patch list is a small
 *            host-side object; it is checked on the host and passed to the
 *            kernel by value, so no device copy is needed)
 * Returns BIT1_ERANGE, with nothing modified, if any row is outside [0, N).
 */
bit1_status bit1_xor_patch(uint8_t *bits, int64_t N, int64_t K,
                           const int32_t *rows, int64_t n_rows,
                           bit1_stream_t stream);

/* Kernels bound every wait on an asynchronous copy; a wait that gives up
 * skips the remaining work and records the event on the device instead of
 * hanging.  Returns how many such events happened since the previous call
 * (and resets the count); synchronises with the device.  0xffffffff if the
 * count could not be read. */
unsigned int bit1_device_wait_timeouts(void);

/* Self-test of that failure path: launches one kernel whose bounded wait is
 * on a barrier that nothing completes.  The wait gives up after a short limit
 * of its own (2^12 polls of a suspending try_wait: milliseconds on B300; the
 * product kernels allow 2^22 polls, about 16 s), the kernel
 * records the event (the next bit1_device_wait_timeouts() is nonzero),
 * writes 1 to the device uint32 *d_done and exits normally; the context
 * stays usable.  No fault, trap or hang is involved.  BIT1_EINVAL on a null
 * or misaligned d_done. */
bit1_status bit1_selftest_wait_timeout(unsigned int *d_done, bit1_stream_t stream);

/* ------------------------------------------------------------------------
 * bit1_gemv_tc_noalloc -- the tensor-core batched product (bit1_gemv_ex with
 * variant BIT1_GEMV_TC) without a caller workspace.  The pages have no
 * counterpart of this call.  It is for callers that cannot allocate device
 * memory around the product: real-time paths that must not enter an
 * allocator (cudaMalloc can block and synchronise the device), and plain C
 * hosts that have no device allocator of their own to size a workspace with.
 *   Scratch: one file-scope device array of BIT1_NOALLOC_SCRATCH_BYTES,
 *   which every GPU that loads the library holds until the process exits.
 *   A batch whose fp16 activations fit in it whole (2 * B * K bytes plus 256
 *   per 64-row chunk, e.g. B = 512 at K = 4096) is staged at once; a larger
 *   one is staged one 64-row chunk at a time, each chunk reusing the array,
 *   so any B with K <= 32768 fits.  Its address is taken with
 *   cudaGetSymbolAddress once per device, on the first call on that device
 *   (a failed lookup is tried again on the next call): make that first call
 *   before any stream capture.
 *   Races: every call on a device uses the same scratch, so two calls whose
 *   kernels overlap on the GPU (different streams, or different host threads
 *   without ordering) corrupt each other's results; keep such calls ordered,
 *   e.g. on one stream.
 * Arguments as bit1_gemv_ex (flags: BIT1_FLAG_PDL, BIT1_FLAG_SWIGLU).
 * Returns BIT1_ESHAPE if
 * the shape is outside the tensor-core kernel's limits (K a multiple of 1024)
 * or needs more scratch than BIT1_NOALLOC_SCRATCH_BYTES (only possible for
 * K > 32768: the need is 2 * min(B, 64) rounded up to 16 * K + 256 bytes,
 * each part rounded up to 256), checked
 * before any CUDA call; BIT1_ECUDA if the scratch address cannot be
 * obtained; otherwise as bit1_gemv_ex.  Allocates nothing.
 */
#define BIT1_NOALLOC_SCRATCH_BYTES ((size_t)4 * 1024 * 1024 + 4096)
bit1_status bit1_gemv_tc_noalloc(const uint8_t *bits, const uint16_t *scales,
                                 const uint16_t *x, int64_t B, int64_t N, int64_t K,
                                 void *y, int y_dtype, unsigned flags,
                                 bit1_stream_t stream);

/* ------------------------------------------------------------------------
 * Ternary weights in 2-bit slots (page "Bonsai 27B: ...", section
 * "삼진(Ternary) 가중치 형식": w = s_g * t with t in {-1, 0, +1} and one FP16
 * scale per 128 inputs; section "저장 공간과 실제 배포 크기": the current
 * kernels keep each ternary value in a 2-bit slot, 2.125 bits/weight with the
 * scales, against the log2(3) + 16/128 ~ 1.71 bits of the ideal code).
 * This library's reading of the slot (the pages do not lay it out): two sign
 * planes a and b, each [N][K/8] in the binary layout above, with
 *     t = (a + b) / 2   (a bit read as +-1):  (1,1) -> +1, (0,0) -> -1,
 *                                             (1,0) and (0,1) -> 0,
 * and one fp16 scale array [N][K/128] shared by both planes.  Flipping a row
 * in both planes with bit1_xor_patch negates that row (0 stays 0); the
 * Bankai page notes that XOR patching does not carry over to ternary codes
 * in general, and this library offers no ternary patch call.
 *
 * bit1_ternary_planes -- codes -> planes: a = (t >= 0), b = (t > 0).
 *   codes   : device, int8 [N][K], each -1, 0 or +1
 *   a, b    : device, N*K/8 bytes each (written)
 *   d_flags : device pointer to one uint32, or NULL.  The call zeroes it on
 *             `stream`; the kernel sets bit 2 if any code is outside
 *             {-1, 0, +1} (the planes are then unspecified).  After
 *             synchronising, bit1_pack_flags_status() maps bit 2 to
 *             BIT1_ERANGE.
 * Returns BIT1_ESHAPE / BIT1_EINVAL on bad arguments (nothing launched),
 * BIT1_ECUDA on launch failure, else BIT1_OK.
 */
bit1_status bit1_ternary_planes(const int8_t *codes, int64_t N, int64_t K,
                                uint8_t *a, uint8_t *b, uint32_t *d_flags,
                                bit1_stream_t stream);

/* bit1_gemv_ternary -- y[b][n] = sum_g s[n][g] * sum_{k in g} t(n,k) x[b][k]
 * for the planes above, computed as the mean of the two binary products
 * (one bit1_gemv_ex pass per plane into fp32 scratch, then one combine
 * kernel).  Result within 1e-3 * sum_k |s*x_k| + 1e-6 of the exact value
 * (plus the bf16 output rounding for y_dtype = BIT1_BF16).
 *   a, b, scales, x, B, N, K, y, y_dtype, variant, flags : as bit1_gemv_ex
 *                  (the variant and BIT1_FLAG_PDL apply to both binary
 *                  passes).  BIT1_FLAG_SWIGLU: rows are interleaved gate/up
 *                  pairs (N even, else BIT1_ESHAPE); both passes run plain
 *                  and the combine writes h = silu(g) * u of the two means,
 *                  [B][N/2], at any batch and with any variant.
 *   workspace    : REQUIRED device scratch of ws_bytes bytes, 16-byte
 *                  aligned: at least the two fp32 halves, 2 * (B*N*4 rounded
 *                  up to 256) bytes, else BIT1_EINVAL; the fastest kernels
 *                  want bit1_gemv_ternary_workspace_bytes(B, N, K).
 * Checks every argument of both passes before launching anything.
 */
size_t bit1_gemv_ternary_workspace_bytes(int64_t B, int64_t N, int64_t K);
bit1_status bit1_gemv_ternary(const uint8_t *a, const uint8_t *b,
                              const uint16_t *scales, const uint16_t *x,
                              int64_t B, int64_t N, int64_t K, void *y,
                              int y_dtype, void *workspace, size_t ws_bytes,
                              int variant, unsigned flags, bit1_stream_t stream);
/* Kernel launches of one bit1_gemv_ternary call (0 on bad arguments). */
int bit1_gemv_ternary_launches(int64_t B, int64_t N, int64_t K, int variant);

/* bit1_ternary_combine -- y[i] = (ya[i] + yb[i]) / 2 for i < n, fp32 sum,
 * output fp32 or bf16 (round to nearest even).  The second step of
 * bit1_gemv_ternary, exposed so that many ternary matrices run as one
 * bit1_gemv_group launch (two problems per matrix, fp32 outputs laid out
 * contiguously) plus one combine.  All pointers device, 16-byte aligned. */
bit1_status bit1_ternary_combine(const float *ya, const float *yb, int64_t n,
                                 void *y, int y_dtype, bit1_stream_t stream);

/* ------------------------------------------------------------------------
 * Ternary codes packed five per byte: a storage closer to the ideal
 * log2(3) bits (same page and sections as above; the pages give no layout).
 * This library's packing: row-major [N][K/128 * 26] bytes; the 128 codes of
 * group g of row n are the 26 bytes at (n * K/128 + g) * 26: byte j < 25
 * holds codes 5j .. 5j+4 and byte 25 holds codes 125 .. 127, each byte the
 * base-3 number v = sum_i (t_i + 1) * 3^i with i = 0 for the lowest k
 * (0 .. 242; the last byte 0 .. 26).  With the fp16 scales [N][K/128] (the
 * same array as the other layouts) this is 1.75 bits/weight, against 2.125
 * for the 2-bit slots.  Flag bits (read with bit1_pack_flags_status, which
 * maps them to BIT1_ERANGE): bit 2 a code outside {-1, 0, +1}, bit 3 a byte
 * outside its range.  d_flags as in bit1_pack: optional, zeroed by the call.
 *
 * bit1_t5_pack      -- codes int8 [N][K] -> packed bytes.
 * bit1_t5_to_planes -- packed bytes -> the two planes of the 2-bit-slot
 *                      layout (N*K/8 bytes each), so a matrix stored in this
 *                      compact form runs on bit1_gemv_ternary's kernels.
 * bit1_gemv_t5      -- y[B][N] straight from the packed bytes, fp32
 *                      accumulation, within the bit1_gemv tolerance.  At
 *                      B = 1 with K a multiple of 1024: a table-lookup
 *                      kernel (a byte splits into v mod 27 and v / 27, each
 *                      looked up in a small table of activation partial
 *                      sums; deterministic).  Otherwise one warp per row, up
 *                      to 8 batch rows per launch (bit1_gemv_t5_launches).
 *                      A byte out of range gives an unspecified (but
 *                      in-bounds) result for its row.
 * All pointers device, 16-byte aligned; BIT1_ESHAPE / BIT1_EINVAL on bad
 * arguments with nothing launched.
 */
bit1_status bit1_t5_pack(const int8_t *codes, int64_t N, int64_t K,
                         uint8_t *packed, uint32_t *d_flags, bit1_stream_t stream);
bit1_status bit1_t5_to_planes(const uint8_t *packed, int64_t N, int64_t K,
                              uint8_t *a, uint8_t *b, uint32_t *d_flags,
                              bit1_stream_t stream);
bit1_status bit1_gemv_t5(const uint8_t *packed, const uint16_t *scales,
                         const uint16_t *x, int64_t B, int64_t N, int64_t K,
                         void *y, int y_dtype, bit1_stream_t stream);
int bit1_gemv_t5_launches(int64_t B, int64_t N, int64_t K);

/* Static description of a status code. */
const char *bit1_status_str(bit1_status status);

/* Library version string. */
const char *bit1_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BIT1_H */
