/*
 * libf8 — Float8 training linear with dynamic tensorwise scaling, for one
 * NVIDIA GB300 (sm_103a).
 *
 * The method (torchtitan's Float8 training, provided by torchao):
 *   "TorchTitan" paper summary (atlas.scime.ai), Approach and the ablation
 *   table — Float8 is applied to the linears of Llama 3.1 8B on top of
 *   torch.compile and FSDP2; wassimseifeddine.com/posts/torchtitan, section
 *   "Float8 Training"; stanleyjacob.dev/oss/torchtitan, Part XI item 9 — the
 *   E4M3 encoding of "FP8 Formats for Deep Learning".  The recipe itself is
 *   not printed on those pages; this library implements the plainest
 *   reading of "dynamic tensorwise scaling":
 *
 *     amax  = max |v| over the whole bf16 tensor                (fp32)
 *     s     = 448 / max(amax, 1e-12)                 (one IEEE fp32 division)
 *     q     = satfinite_rne_e4m3(fl32(v * s))          (byte per element)
 *     Y  = bf16( (q(X)  q(W)^T)  / (s_x  s_w) )        forward
 *     dX = bf16( (q(dY) q(W))    / (s_dy s_w) )        dgrad
 *     dW = bf16( (q(dY)^T q(X))  / (s_dy s_x) )        wgrad
 *   with the products accumulated in fp32 on the tensor cores.
 *
 * Conventions for every call:
 *   - Tensors are dense and row-major.  X is [M,K] (tokens x in-features),
 *     W is [N,K] (nn.Linear layout), dY and Y are [M,N], dX is [M,K], dW is
 *     [N,K].  bf16 tensors are passed as `const void*`; E4M3 tensors as
 *     `uint8_t*` holding float8_e4m3fn codes.
 *   - Every pointer is a DEVICE pointer of the current CUDA device, owned by
 *     the caller.  The library allocates nothing per call.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on it and returns; scales and amax values stay
 *     in device memory and are never read back by the library.
 *   - Argument errors are found on the host before anything is launched and
 *     are returned as a non-zero f8_status; nothing is enqueued then.
 *     Pointers to bf16 or E4M3 tensors must be 16-byte aligned; pointers to
 *     fp32 scalars 4-byte aligned.
 *   - Errors found on the device (a non-finite amax, a wait that ran past its
 *     time limit, in the checked build an index outside its buffer) are
 *     recorded in a per-device status word;
 *     f8_last_device_status() reports and clears it.
 */
#ifndef F8_H_
#define F8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    F8_OK = 0,
    F8_ERR_INVALID = 1,     /* NULL pointer, negative size, bad combination   */
    F8_ERR_ALIGN = 2,       /* a pointer is not 16-byte (tensors) / 4-byte aligned */
    F8_ERR_SHAPE = 3,       /* a size breaks a layout rule (e.g. K % 16 != 0) */
    F8_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed           */
    F8_ERR_TIMEOUT = 5,     /* a device-side wait exceeded its time limit     */
    F8_ERR_NONFINITE = 6,   /* an amax input held +-inf or NaN                */
    F8_ERR_UNSUPPORTED = 7, /* not an sm_103 device, or no driver entry point */
    F8_ERR_BOUNDS = 8       /* checked build only: an index left its buffer   */
} f8_status;

/*
 * FP8 formats of "FP8 Formats for Deep Learning" (the paper the torchtitan
 * walkthrough, Part XI item 9, cites for torchtitan's Float8 training):
 *   F8_E4M3  1-4-3, bias 7, no infinities, largest finite 448;
 *   F8_E5M2  1-5-2, bias 15, IEEE-style inf/NaN, largest finite 57344.
 * The five calls of the path use E4M3 for X, W and dY; the _fmt variants
 * below also take E5M2, the wider-range format the paper suggests for
 * gradients.  Scales are then fmax / max(amax, 1e-12), fmax the format's
 * largest finite value, and conversions saturate to +-fmax.
 */
typedef enum { F8_E4M3 = 0, F8_E5M2 = 1 } f8_format;

/*
 * Step 1 of dynamic tensorwise scaling: the tensor's absolute maximum.
 * Source: wassimseifeddine.com/posts/torchtitan, section "Float8 Training"
 * (torchtitan's Float8 is torchao's Float8 training) and the atlas summary
 * of the TorchTitan paper, Approach (Float8 is one of the composable
 * training transformations).  The pages name neither the scaling recipe nor
 * an interface; amax over the whole tensor is the plainest reading of
 * "dynamic tensorwise" scaling, and this call is this library's own.
 *
 * amax_out[0] = max_i |x[i]| over n bf16 values, as fp32 (exact).
 *   x:        device, n bf16 values, 16-byte aligned.  n == 0 gives 0.
 *   amax_out: device, one fp32; overwritten (the call zeroes it first).
 * A NaN or +-inf input sets F8_ERR_NONFINITE in the device status word; the
 * value written is then unspecified.
 */
f8_status f8_amax(const void *x, int64_t n, float *amax_out, void *stream);

/*
 * Steps 2 and 3 of dynamic tensorwise scaling: the scale and the cast.
 * Source: stanleyjacob.dev/oss/torchtitan, Part XI (reading list), item 9:
 * torchtitan's Float8 uses the E4M3 encoding of "FP8 Formats for Deep
 * Learning" (largest finite value 448, no infinities); the scale that maps
 * amax onto 448 and the saturating round-to-nearest-even conversion follow
 * from that format.  The pages print no interface; emitting both layouts
 * in one pass is this library's design (the backward GEMMs take the
 * transposed copy as a K-major operand).
 *
 * Scale and cast one bf16 tensor to E4M3, emitting both layouts in one pass.
 *   x:          device bf16 [rows, cols], 16-byte aligned.
 *   amax:       device fp32 scalar (e.g. from f8_amax).
 *   scale_out:  device fp32 scalar receiving s = 448 / max(amax, 1e-12), or NULL.
 *   q:          device uint8 [rows, cols] (row-major copy) or NULL.
 *   q_t:        device uint8 [cols, rows] (column-major copy: q_t[c*rows + r]
 *               == q[r*cols + c]) or NULL.
 * Each element is q = satfinite_rne_e4m3(fl32(x * s)): one fp32 multiply,
 * then round-to-nearest-even onto the E4M3 grid, |v| >= 448 -> +-448.
 * Any rows, cols >= 0 are accepted; shapes with rows % 16 == 0 and
 * cols % 16 == 0 take the vectorised path.
 */
f8_status f8_cast_transpose(const void *x, int64_t rows, int64_t cols, const float *amax,
                            float *scale_out, uint8_t *q, uint8_t *q_t, void *stream);

/*
 * f8_amax followed by f8_cast_transpose as two back-to-back launches with
 * nothing in between: the amax launch leaves one partial maximum per CTA in
 * `workspace` (so no output has to be zeroed first), the cast launch reduces
 * them in its prologue, writes amax_out and scale_out, and casts; its re-read
 * of the tensor comes mostly from L2.  Results are bit-identical to the two
 * separate calls.  This is the quantisation f8_linear_fwd/bwd perform.
 *   x:          device bf16 [rows, cols], 16-byte aligned.
 *   amax_out:   device fp32 scalar receiving max |x|.
 *   scale_out:  device fp32 scalar receiving s = 448 / max(amax, 1e-12), or NULL.
 *   q, q_t:     as for f8_cast_transpose (either may be NULL).
 *   workspace:  device scratch of f8_quantize_workspace_bytes() bytes,
 *               16-byte aligned; its contents need not be initialised and
 *               are meaningless after the call.  Two calls whose GPU work
 *               overlaps must not share one workspace.
 * A non-finite input sets F8_ERR_NONFINITE in the device status word.
 */
size_t f8_quantize_workspace_bytes(void);
f8_status f8_quantize(const void *x, int64_t rows, int64_t cols, float *amax_out,
                      float *scale_out, uint8_t *q, uint8_t *q_t, void *workspace,
                      size_t workspace_bytes, void *stream);

/* f8_quantize into format `fmt` (E4M3: identical to f8_quantize). */
f8_status f8_quantize_fmt(const void *x, int64_t rows, int64_t cols, f8_format fmt,
                          float *amax_out, float *scale_out, uint8_t *q, uint8_t *q_t,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Dynamic tensorwise quantisation of several tensors at once, each with its
 * own amax and scale: every tensor gets exactly what f8_quantize_fmt gives
 * it (bit-identical).  Consecutive tensors whose sides are multiples of 128
 * share a launch pair while their bf16 total stays within 112 MiB (one
 * amax launch whose CTAs are split between the tensors in proportion to
 * their sizes, then one TMA cast launch over all their 128 x 128 tiles; the
 * cast's re-read then still finds the amax pass's reads in L2); a larger
 * tensor, or one with other sides, gets f8_quantize_fmt's pair of its own.
 * Two launches instead of two per tensor matter for the small tensors of a
 * step (the 8-33 MB weights of the Llama-3.1-8B attention projections),
 * whose launches are dominated by ramp-up rather than bytes: e.g. all the
 * weights of a model once per optimiser step, or the dY of linears that
 * share an input.
 *   tensors: host array of `count` (1 .. F8_MAX_MULTI_TENSORS) entries;
 *            x, amax_out required, scale_out, q, q_t may be NULL; pointers
 *            aligned as for f8_quantize.
 *   fmt:     the format of every tensor of the call (F8_E4M3 or F8_E5M2).
 *   workspace: f8_quantize_multi_workspace_bytes() bytes, 16-byte aligned,
 *            contents need not be initialised.
 * The scaling recipe is the one above (atlas summary Approach: Float8 as a
 * per-linear transformation; one scale per tensor).  The pages print no
 * interface for it.
 */
#define F8_MAX_MULTI_TENSORS 8
typedef struct {
    const void *x;          /* device bf16 [rows, cols] */
    int64_t rows, cols;
    float *amax_out;        /* device fp32 scalar receiving max |x| */
    float *scale_out;       /* device fp32 scalar receiving the scale, or NULL */
    uint8_t *q;             /* device codes [rows, cols] or NULL */
    uint8_t *q_t;           /* device codes [cols, rows] or NULL */
} f8_quant_tensor;
size_t f8_quantize_multi_workspace_bytes(void);
f8_status f8_quantize_multi(const f8_quant_tensor *tensors, int count, f8_format fmt,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Step 4 of the Float8 linear: the FP8 GEMM with the inverse-scale epilogue.
 * Source: the discuss.pytorch.org torchtitan index, topic "[Distributed w/
 * Torchtitan] Enabling Float8 All-Gather in FSDP2" (float8 speeds up large
 * GEMMs), and the atlas summary's ablation table (Float8 on Llama 3.1 8B).
 * Dividing the fp32 accumulator by the two scales undoes the scaling of
 * the casts; the pages print no interface and no kernel.
 *
 * C = bf16( A B^T / (scale_a * scale_b) ), fp32 accumulation on tcgen05.
 *   a:       device E4M3 [M, K] row-major (K contiguous), 16-byte aligned.
 *   b:       device E4M3 [N, K] row-major (K contiguous), 16-byte aligned.
 *   scale_a, scale_b: device fp32 scalars (the scales the operands were cast with).
 *   c:       device bf16 [M, N] row-major, 16-byte aligned; fully overwritten.
 * K must be a multiple of 16 (the E4M3 row pitch must be a multiple of 16
 * bytes); M, N >= 0 are otherwise free.  K == 0 writes zeros.
 */
f8_status f8_gemm(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                  const float *scale_a, const float *scale_b, void *c, void *stream);

/* f8_gemm with the operands' formats given (any mix of E4M3 and E5M2; one
 * tcgen05.mma kind::f8f6f4 takes both). */
f8_status f8_gemm_fmt(const uint8_t *a, f8_format fmt_a, const uint8_t *b, f8_format fmt_b,
                      int64_t M, int64_t N, int64_t K, const float *scale_a,
                      const float *scale_b, void *c, void *stream);

/*
 * One GEMM of f8_gemm_grouped: c = bf16( a b^T / (scale_a * scale_b) ),
 * with the arguments of f8_gemm_fmt.
 */
typedef struct {
    const uint8_t *a;       /* device [M, K], K contiguous, format fmt_a */
    const uint8_t *b;       /* device [N, K], K contiguous, format fmt_b */
    int64_t M, N, K;
    const float *scale_a;   /* device fp32 scalars */
    const float *scale_b;
    void *c;                /* device bf16 [M, N] row-major */
    f8_format fmt_a, fmt_b;
} f8_gemm_problem;

/*
 * `count` (1 .. F8_MAX_GROUPED_GEMMS) independent GEMMs in as few
 * persistent launches as pay.  A launch takes up to four problems whose K
 * extents take at most two values; their tiles share the CTA pairs under a
 * static list schedule: the problems with more K per tile are dealt
 * round-robin, then the others' tiles go in order to whichever pair frees
 * up first, so one problem's last, partial wave is filled with another's
 * tiles.  A planner splits the problems into launches and shares a launch
 * only where its predicted time beats one launch per problem by 4%.  Each
 * c is bit-identical to f8_gemm_fmt on its problem (same tiles, same K
 * order).  f8_linear_bwd runs its dgrad and wgrad GEMMs this way (the two
 * products of the Float8 linear's backward pass, both reading q(dY)), and
 * f8_linear_fwd_group / f8_linear_bwd_group the GEMMs of linears that
 * share their input.
 *   problems: host array of `count` problems, each checked as by
 *   f8_gemm_fmt (F8_ERR_INVALID for count outside 1..F8_MAX_GROUPED_GEMMS
 *   or a NULL array).  The c buffers must not overlap one another or any
 *   operand.
 * Problems that need different kernels (M < 256 for one, M >= 256 for
 * another) or have a zero extent run as separate launches, in array order.
 * The pages print no interface; the call exists because several GEMMs of
 * one step are independent (the linear's own dgrad and wgrad; the q, k and
 * v projections that share X in the Llama 3.1 block of the atlas summary's
 * ablation table).
 */
#define F8_MAX_GROUPED_GEMMS 8
f8_status f8_gemm_grouped(const f8_gemm_problem *problems, int count, void *stream);

/*
 * What the forward pass leaves for the backward pass.  All members are
 * caller-allocated device buffers.
 *   x_t [K, M], w_t [K, N]: E4M3 column-major copies of q(X) and q(W);
 *   amax_x, scale_x, amax_w, scale_w: device fp32 scalars.
 */
typedef struct {
    uint8_t *x_t;
    uint8_t *w_t;
    float *amax_x;
    float *scale_x;
    float *amax_w;
    float *scale_w;
} f8_linear_saved;

/*
 * Device workspace (bytes) that f8_linear_fwd and f8_linear_bwd need for
 * (M, N, K): the row-major E4M3 copies of X and W (forward) or of dY and
 * dY^T plus two scalars (backward), and the per-CTA partial maxima of the
 * amax launches; each region 256-byte aligned.  Its contents need not be
 * initialised.
 */
size_t f8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Forward of a Float8 linear.  Source: the atlas summary of the TorchTitan
 * paper, Approach (Float8 applied to the model's linears as a composable
 * transformation) and the ablation table's rows "add Float8 on top of
 * torch.compile" (Llama 3.1 8B, 8 and 128 GPUs); wassimseifeddine.com,
 * "Float8 Training".  Its steps are those of f8_amax, f8_cast_transpose and
 * f8_gemm above on X and W; the pages print no interface.
 *
 * Y [M,N] = X [M,K] W[N,K]^T.
 *   x, w: device bf16 inputs; y: device bf16 output.
 *   saved: filled with q(X)^T, q(W)^T and the four scalars.
 *   workspace: device scratch of at least f8_linear_workspace_bytes(M,N,K)
 *   bytes, 256-byte aligned; its contents are not needed after the call.
 * M, N, K must be multiples of 16 and > 0.
 */
f8_status f8_linear_fwd(const void *x, const void *w, int64_t M, int64_t N, int64_t K, void *y,
                        const f8_linear_saved *saved, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * Backward of a Float8 linear.  Source: as f8_linear_fwd (the atlas
 * summary's Approach and ablation table: Float8 training of the linears,
 * so their gradients too run as FP8 GEMMs); the pages print no interface.
 *
 * Backward of the same linear: dX [M,K] = dY W, dW [N,K] = dY^T X, using the
 * saved q(X)^T, q(W)^T and scales from f8_linear_fwd (which must have been
 * enqueued earlier on the same stream, or otherwise completed).  dY is
 * quantised (amax launch, cast launch), then both GEMMs run as one launch
 * (f8_gemm_grouped).
 *   dy: device bf16 [M,N]; dx, dw: device bf16 outputs (either may be NULL
 *   to skip that GEMM).  Workspace as for the forward pass.
 */
f8_status f8_linear_bwd(const void *dy, const f8_linear_saved *saved, int64_t M, int64_t N,
                        int64_t K, void *dx, void *dw, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * f8_linear_fwd for callers that cannot allocate device memory.  (The
 * pages describe no such call; it exists for this library's users.)
 *
 * Who needs it: code that may not call cudaMalloc, such as a plugin running
 * inside a framework that owns all device memory through its own pool and
 * forbids side allocations, or a service whose device-memory budget is fixed
 * at start-up.  Such a caller cannot supply f8_linear_fwd's workspace.
 *
 * What it does: exactly what f8_linear_fwd does (the same code, kernels and
 * arguments), except that the workspace is a static device array of
 * F8_NOALLOC_SCRATCH_BYTES compiled into the library.  The caller still
 * passes x, w, y and `saved`.  The call allocates nothing and calls no
 * allocating routine.
 *
 * Limits and rules:
 *  - f8_linear_fwd's workspace for (M, N, K) must fit in
 *    F8_NOALLOC_SCRATCH_BYTES (64 MiB): the E4M3 copies of X and W, M*K +
 *    N*K bytes each rounded up to 256, plus 32 KiB of partial maxima.
 *    Larger problems return F8_ERR_SHAPE before anything is launched.
 *    M, N, K: multiples of 16, > 0.
 *  - Every device that loads the library holds the array until the process
 *    exits.
 *  - All calls share the array.  Calls whose GPU work overlaps (different
 *    streams, or threads without ordering between them) race on it and may
 *    produce wrong results; calls on one stream are safe.
 *  - The first call on a device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 */
#define F8_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
f8_status f8_linear_fwd_noalloc(const void *x, const void *w, int64_t M, int64_t N, int64_t K,
                                void *y, const f8_linear_saved *saved, void *stream);

/*
 * Linears that read one input X (in the Llama 3.1 block the q, k and v
 * projections, and w1 and w3 of the FFN), each a Float8 linear of its own
 * (atlas summary, Approach: Float8 is a per-linear transformation): X is
 * quantised once with one scale, every weight W_i with its own scale, and
 * every output is bit-identical to f8_linear_fwd / f8_linear_bwd_fmt on
 * that member with the same X.  One member of the group:
 *   N:     out-features of this linear (multiple of 16, > 0);
 *   w:     forward: device bf16 W_i [N, K];  y: device bf16 Y_i [M, N];
 *   dy:    backward: device bf16 dY_i [M, N];
 *   dx:    backward: device bf16 dX_i [M, K] or NULL (this member's own
 *          share; the caller sums the members' dX if the model does);
 *   dw:    backward: device bf16 dW_i [N, K] or NULL;
 *   saved: as for f8_linear_fwd.  x_t, amax_x and scale_x must be the same
 *          buffers in every member (the group's one q(X)^T and X scalars,
 *          written once); w_t, amax_w, scale_w are the member's own.
 */
#define F8_MAX_GROUP_LINEARS 4
typedef struct {
    int64_t N;
    const void *w;
    void *y;
    const void *dy;
    void *dx;
    void *dw;
    f8_linear_saved saved;
} f8_group_linear;

/*
 * Device workspace (bytes) f8_linear_fwd_group and f8_linear_bwd_group need
 * for M, K and the members' N (count of them); 256-byte aligned regions,
 * contents need not be initialised.  0 for bad arguments.
 */
size_t f8_linear_group_workspace_bytes(int64_t M, int64_t K, const int64_t *N, int count);

/*
 * Forward of a group of `count` (1 .. F8_MAX_GROUP_LINEARS) linears sharing
 * X [M, K]: Y_i = X W_i^T.  Launches: X and every W_i quantised together
 * (f8_quantize_multi: two launches; per tensor where a side is not a
 * multiple of 128), then the count GEMMs under f8_gemm_grouped's planner:
 * with one K they form one class, and one launch runs all their tiles
 * round-robin where that is predicted to pay (the skinny k and v
 * projections, 128 tiles of 256 x 256 each at M = 8192, no longer run as
 * launches of 1.7 waves).
 *   members: host array; uses N, w, y, saved.  M, K multiples of 16, > 0.
 */
f8_status f8_linear_fwd_group(const void *x, int64_t M, int64_t K, const f8_group_linear *members,
                              int count, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward of the same group: every dY_i quantised in format fmt_dy
 * (f8_quantize_multi), then every member's dgrad dX_i = dY_i W_i and wgrad
 * dW_i = dY_i^T X (up to 2 x count GEMMs) under f8_gemm_grouped's planner.
 *   members: host array; uses N, dy, dx, dw, saved (from the forward,
 *   enqueued earlier on the same stream or completed).
 */
f8_status f8_linear_bwd_group(const f8_group_linear *members, int count, int64_t M, int64_t K,
                              f8_format fmt_dy, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * The FP8 weight all-gather of FSDP2 (the discuss.pytorch.org torchtitan
 * index, topic "[Distributed w/ Torchtitan] Enabling Float8 All-Gather in
 * FSDP2": float8 saves network bandwidth with reduced message size).  Each
 * rank holds a row shard of W; the ranks agree on one tensorwise scale
 * (all-reduce MAX of the shards' amax), cast their shard with it and
 * all-gather the E4M3 bytes, half the bytes of a bf16 gather.  The
 * collectives themselves are the caller's (float8_mixed_precision_gb300.fsdp
 * issues them with torch.distributed); these two calls are the device steps
 * that the gathered weight then needs.  The pages print no interface.
 *
 * f8_transpose_u8: out[c, r] = in[r, c] for a [rows, cols] byte tensor
 * (device pointers, no alignment rule, rows, cols >= 0; not in place).  It
 * makes q(W)^T [K, N], the dgrad operand, from the gathered q(W) [N, K].
 * With rows and cols multiples of 128 and both pointers 16-byte aligned it
 * moves 16-byte vectors through 128 x 128 tiles; otherwise it moves bytes.
 */
f8_status f8_transpose_u8(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out,
                          void *stream);

/*
 * Forward of a Float8 linear whose weight arrives already quantised (the
 * gathered q(W) above): X is quantised as in f8_linear_fwd (amax launch,
 * cast launch), then Y = bf16(q(X) q(W)^T / (s_x s_w)).
 *   w_q:   device E4M3 [N, K], the row-major q(W).
 *   saved: x_t, amax_x, scale_x are written; w_t, amax_w, scale_w are read
 *          only and must already hold q(W)^T [K, N] and W's scalars (the
 *          scale W was cast with), so f8_linear_bwd applies unchanged.
 *   workspace: f8_linear_fwd_qw_workspace_bytes(M, K) bytes, 256-aligned.
 * Outputs are bit-identical to f8_linear_fwd on the bf16 W whose
 * quantisation q(W) is.
 */
size_t f8_linear_fwd_qw_workspace_bytes(int64_t M, int64_t K);
f8_status f8_linear_fwd_qw(const void *x, const uint8_t *w_q, int64_t M, int64_t N, int64_t K,
                           void *y, const f8_linear_saved *saved, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * f8_linear_bwd with dY quantised to `fmt_dy` (E5M2: scale 57344/amax(dY);
 * dgrad and wgrad then run E5M2 x E4M3 GEMMs).  X and W stay E4M3.
 */
f8_status f8_linear_bwd_fmt(const void *dy, f8_format fmt_dy, const f8_linear_saved *saved,
                            int64_t M, int64_t N, int64_t K, void *dx, void *dw, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * The w2 input of a SwiGLU FFN, h = bf16(silu(a) * b), produced and
 * quantised to E4M3 with its amax taken in the producing pass: launch one
 * reads a and b, writes h and one partial maximum of |h| per CTA; launch two
 * is f8_quantize's cast of h.  Against forming h separately and then
 * running f8_quantize, the amax re-read of h (2 B/elem) is gone.
 * h is the bf16 of silu(a) b with silu(a) = a / (1 + exp(-a)), evaluated
 * in fp32 (exp by Cody-Waite range reduction and the degree-7 Taylor
 * polynomial, the reciprocal correctly rounded): within one bf16 ulp of
 * the exact value rounded once, and equal to it except where the exact
 * value lies within a few fp32 ulp of a bf16 rounding boundary.  The pages
 * name the SwiGLU FFN of torchtitan's Llama 3.1 and credit Float8 on top
 * of torch.compile, which fuses such neighbouring elementwise work.
 *   a, b:     device bf16 [rows, cols], 16-byte aligned.
 *   h:        device bf16 [rows, cols] receiving h.
 *   amax_out, scale_out, q, q_t, workspace: as for f8_quantize.
 */
f8_status f8_quantize_swiglu(const void *a, const void *b, void *h, int64_t rows, int64_t cols,
                             float *amax_out, float *scale_out, uint8_t *q, uint8_t *q_t,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * f8_linear_fwd of the w2 linear fed by h = silu(a) * b (a, b, h: device
 * bf16 [M, K]; h receives the product): the input is produced and quantised
 * by f8_quantize_swiglu's two launches.  `saved` receives q(h)^T, so
 * f8_linear_bwd applies unchanged.
 */
f8_status f8_linear_fwd_swiglu(const void *a, const void *b, void *h, const void *w, int64_t M,
                               int64_t N, int64_t K, void *y, const f8_linear_saved *saved,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * The input side of a SwiGLU FFN (the FeedForward of torchtitan's Llama 3.1:
 * w2(silu(w1(x)) * w3(x))) as one Float8 linear whose GEMM epilogue also
 * forms the w2 input and its amax:
 *   AB = bf16(q(X) q(W13)^T / (s_x s_w13)), the Float8 linear of the group
 *        {w1, w3} that shares X (one tensorwise scale over W13, as for every
 *        concatenated weight);
 *   h  = bf16(silu(a) * b), formed in the epilogue from the bf16 a and b just
 *        rounded, with silu as in f8_quantize_swiglu;
 *   amax(h) taken in the same epilogue (one partial per CTA), then h cast to
 *        E4M3 with both copies.
 * Against f8_linear_fwd on W13 followed by f8_quantize_swiglu, a and b are
 * not read back (4 B per element of h) and the SiLU arithmetic runs under
 * the GEMM's main loop.  Launches: amax and cast of X, amax and cast of W13,
 * the GEMM, the cast of h.
 *   x:     device bf16 [M, K].
 *   w13:   device bf16 [2F, K], W1 and W3 interleaved by 128 rows: rows
 *          [256j, 256j + 128) are W1 rows [128j, 128j + 128) and rows
 *          [256j + 128, 256j + 256) are W3 rows [128j, 128j + 128).
 *          F % 128 == 0, K % 16 == 0, M % 16 == 0.
 *   ab:    device bf16 [M, 2F] receiving a and b, interleaved like W13 (a
 *          tensor of the forward kept for the SwiGLU backward).
 *   h:     device bf16 [M, F] receiving h.
 *   saved: receives q(X)^T, q(W13)^T, their amax and scales, as f8_linear_fwd
 *          with N = 2F does, so f8_linear_bwd (N = 2F, dY interleaved like
 *          AB) is the group's backward.
 *   amax_h, scale_h: device fp32 scalars receiving h's amax and scale.
 *   h_q:   device E4M3 [M, F], q(h) row-major: the A operand of the w2 GEMM
 *          (f8_gemm(h_q, q(W2), ..., scale_h, s_w2)).
 *   h_t:   device E4M3 [F, M], q(h)^T: the w2 linear's saved input.
 *   workspace: f8_linear_workspace_bytes(M, 2F, K) bytes, 256-byte aligned.
 * All device pointers 16-byte aligned (amax_h, scale_h: 4).  F8_ERR_SHAPE
 * if F is not a positive multiple of 128.
 */
f8_status f8_linear_fwd_w13_swiglu(const void *x, const void *w13, int64_t M, int64_t F,
                                   int64_t K, void *ab, void *h, const f8_linear_saved *saved,
                                   float *amax_h, float *scale_h, uint8_t *h_q, uint8_t *h_t,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * The first half of f8_linear_bwd_w13_swiglu alone: d(AB) from dh and the
 * forward's AB with its amax (one pass), then its E4M3 cast, as
 * f8_quantize does for a given tensor.
 *   dh:  device bf16 [M, F]; ab: device bf16 [M, 2F]; F % 128 == 0.
 *   dab: device bf16 [M, 2F] receiving d(AB).
 *   fmt: F8_E4M3 or F8_E5M2 (as f8_quantize_fmt).
 *   amax_out, scale_out, q ([M, 2F]), q_t ([2F, M]), workspace
 *   (f8_quantize_workspace_bytes()): as for f8_quantize.
 */
f8_status f8_quantize_swiglu_bwd(const void *dh, const void *ab, int64_t M, int64_t F, void *dab,
                                 f8_format fmt, float *amax_out, float *scale_out, uint8_t *q,
                                 uint8_t *q_t, void *workspace, size_t workspace_bytes,
                                 void *stream);

/*
 * The backward of f8_linear_fwd_w13_swiglu for the gradient dh of h (in a
 * Llama FFN, the dX of the w2 linear):
 *   d(AB) = the gradient of h = silu(a) * b: db = bf16(dh * silu(a)),
 *           da = bf16(dh * b * silu'(a)) with silu'(a) = sigma (1 + a (1 -
 *           sigma)), in fp32 as in the forward and to the same bound (one
 *           bf16 ulp of the exact value); written in AB's column order, with
 *           its amax taken in the same pass (one partial per CTA);
 *   then the group's backward as f8_linear_bwd with dY = d(AB): cast of
 *           d(AB), dX = q(dAB) q(W13), dW13 = q(dAB)^T q(X).
 *   dh:    device bf16 [M, F].
 *   ab:    device bf16 [M, 2F], the forward's AB.
 *   saved: the forward's saved tensors.
 *   dab:   device bf16 [M, 2F] receiving d(AB).
 *   fmt_dab: F8_E4M3, or F8_E5M2 for the E5M2-gradient recipe (d(AB) cast
 *          with scale 57344/amax; E5M2 x E4M3 GEMMs), as f8_linear_bwd_fmt.
 *   dx:    device bf16 [M, K] or NULL; dw13: device bf16 [2F, K] or NULL.
 *   workspace: f8_linear_workspace_bytes(M, 2F, K) bytes, 256-byte aligned.
 * All device pointers 16-byte aligned.  F8_ERR_SHAPE if F is not a positive
 * multiple of 128.
 */
f8_status f8_linear_bwd_w13_swiglu(const void *dh, const void *ab, const f8_linear_saved *saved,
                                   int64_t M, int64_t F, int64_t K, void *dab, f8_format fmt_dab,
                                   void *dx, void *dw13, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * The GEMM of f8_linear_fwd_w13_swiglu alone, for callers that quantise X
 * and W13 themselves (e.g. a W13 quantised once per optimiser step):
 * AB = bf16(q(X) q(W13)^T / (scale_x scale_w13)) and h = bf16(silu(a) * b)
 * from the epilogue, with max |h| written to amax_h.
 *   x_q:   device E4M3 [M, K]; w13_q: device E4M3 [2F, K], rows interleaved
 *          as for f8_linear_fwd_w13_swiglu; F % 128 == 0, M % 16 == 0,
 *          K % 16 == 0.
 *   scale_x, scale_w13: device fp32 scalars.
 *   ab:    device bf16 [M, 2F]; h: device bf16 [M, F].
 *   amax_h: device fp32, zeroed by this call (a 4-byte memset on `stream`)
 *          and then raised by one atomicMax per CTA; it is ready for
 *          f8_cast_transpose(h, ...).  A non-finite h sets F8_ERR_NONFINITE.
 */
f8_status f8_gemm_w13_swiglu(const uint8_t *x_q, const uint8_t *w13_q, int64_t M, int64_t F,
                             int64_t K, const float *scale_x, const float *scale_w13, void *ab,
                             void *h, float *amax_h, void *stream);

/*
 * Number of kernels this library has launched (enqueued) in this process so
 * far, over all devices and streams; host-side, no synchronisation.  The
 * difference across a sequence of calls is the number of GPU kernels those
 * calls launched (memsets are not counted).
 */
unsigned long long f8_kernel_launches(void);

/*
 * The checked build (compiled with -DF8_BOUNDS_CHECK) tests every manually
 * indexed global load and store of the amax, cast and SwiGLU kernels and of
 * the GEMM's direct-store epilogue against its buffer before making it; an
 * index outside the buffer skips the access and sets F8_ERR_BOUNDS in the
 * device status word (in place of a sanitizer, which this build does not
 * rely on).  f8_selftest_bounds launches one thread that makes one such
 * check fail without touching memory: in the checked build it returns F8_OK
 * and the next f8_last_device_status() gives F8_ERR_BOUNDS; in a release
 * build it launches nothing and returns F8_ERR_UNSUPPORTED.
 */
f8_status f8_selftest_bounds(void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns F8_OK, F8_ERR_NONFINITE, F8_ERR_TIMEOUT or F8_ERR_BOUNDS
 * (the most severe bit set, BOUNDS over TIMEOUT over NONFINITE), or
 * F8_ERR_CUDA if the synchronisation itself failed.
 */
f8_status f8_last_device_status(void *stream);

/* Static, human-readable name of a status code. */
const char *f8_status_string(f8_status status);

/*
 * Failure-path self-test: launches one CTA that waits on an mbarrier nothing
 * ever arrives on, using the same bounded wait as the GEMM pipeline, with a
 * limit of `limit_ns` nanoseconds.  The wait gives up, records
 * F8_ERR_TIMEOUT in the status word and the kernel returns normally, so the
 * context stays usable.  Read the result with f8_last_device_status().
 */
f8_status f8_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/*
 * Time limit (nanoseconds) of every device-side wait of the GEMM pipeline;
 * default 2e9.  A wait that exceeds it aborts its CTA cleanly and records
 * F8_ERR_TIMEOUT.  0 restores the default.
 */
void f8_set_wait_limit_ns(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* F8_H_ */
