/*
 * ep.h -- C ABI of a single-GPU MoE token dispatch / combine library for
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow the DeepEP pages this library is built from:
 *  - "Redundant atomics in internode_ll" (DeepEP issue #282), the quoted
 *    low-latency dispatch excerpt: a token count per expert, and expert e
 *    living on partition e / (experts per partition) as local expert
 *    e % (experts per partition).
 *  - "Reasons for not calling NVSHMEM public APIs?" (DeepEP issue #18), the
 *    answer on low-latency mode: data for one expert keeps its order.
 *  - "Pipeline direct NVLink dispatch with triple-buffered prefetch" (DeepEP
 *    PR #693), Summary: each token carries hidden data, scale factors,
 *    metadata and routing; the next token is prefetched while earlier stores
 *    drain.  Validation table: dispatch and combine are the measured pair.
 * Here all experts live in one GPU's HBM; partitions are logical only.
 *
 * Conventions for every entry point
 *  - Device pointers are raw CUDA device addresses.  The caller allocates and
 *    frees every buffer (including the layout workspace); the library never
 *    allocates, frees or synchronises.
 *  - All work is enqueued on `stream` (NULL = the legacy default stream).  A
 *    return of EP_OK means the work was enqueued; results are ready once the
 *    stream reaches that point.  Calls are stateless and thread-safe.
 *  - Most kernels launch with programmatic stream serialization and let the
 *    next kernel of the stream start early: each waits for the previous
 *    kernel to complete before it writes memory or reads what that kernel may
 *    write (before the wait it only prefetches into L2).  A caller's kernel
 *    that follows and is itself launched programmatically must likewise
 *    execute griddepcontrol.wait (cudaGridDependencySynchronize) before it
 *    reads this library's outputs; kernels launched normally need nothing.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns EP_ERR_INVALID_ARG (unsupported sizes EP_ERR_UNSUPPORTED)
 *    with nothing enqueued.  A failed launch returns EP_ERR_CUDA.  The text of
 *    the last failure on the calling thread is available from ep_last_error().
 *  - Conditions found on the device never trap: they are OR-ed into the
 *    caller's 32-bit `err_flags` word (EP_ERRF_*), which the caller clears and
 *    reads back.  `err_flags` may be NULL, in which case they are dropped.
 *  - A buffer of zero elements may be passed as NULL.
 *  - Element types: bf16 is stored as 16-bit IEEE bfloat16; fp8 as one byte of
 *    OCP e4m3 ("e4m3fn": bias 7, max 448, no infinities); f32 / i32 native.
 *  - All arrays are dense and row-major.
 */
#ifndef EP_GB300_H_
#define EP_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *ep_stream_t;

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,   /* null or misaligned pointer, bad shape       */
    EP_ERR_UNSUPPORTED = 2,   /* valid but beyond this library's limits, or no
                                 sm_103 device current                        */
    EP_ERR_CUDA = 3           /* a CUDA runtime call or launch failed         */
} ep_status_t;

typedef enum {
    EP_LAYOUT_PACKED = 0,     /* R = T*k rows, expert e owns rows
                                 [offsets[e], offsets[e+1])                   */
    EP_LAYOUT_CAPACITY = 1    /* R = E*capacity rows, expert e owns rows
                                 [e*capacity, (e+1)*capacity)                 */
} ep_layout_mode_t;

/* Payload format of ep_dispatch. */
typedef enum {
    EP_PAYLOAD_BF16 = 0,      /* recv is bf16 [R, H], a bit copy of x         */
    EP_PAYLOAD_FP8_E4M3 = 1,  /* recv is e4m3 [R, H] plus f32 scales [R, H/128] */
    EP_PAYLOAD_FP8_E4M3_UE8M0 = 2 /* e4m3 [R, H] plus power-of-two scales stored
                                 as u8 biased exponents [R, H/128] (UE8M0:
                                 scale = 2^(e - 127))                          */
} ep_payload_t;

/* Bits of the device error word. */
enum {
    EP_ERRF_BAD_EXPERT = 1u,  /* a topk_idx entry outside [-1, E); treated as -1 */
    EP_ERRF_CAPACITY = 2u,    /* capacity mode dropped at least one copy      */
    EP_ERRF_TIMEOUT = 4u,     /* an internal bounded wait ran out; outputs of
                                 that call are incomplete                     */
    EP_ERRF_BAD_SLOT = 8u     /* a slot_of entry >= R (or < -1); that copy was
                                 skipped                                      */
};

/* Limits of this library. */
#define EP_MAX_EXPERTS 1024
#define EP_MAX_TOPK 32

typedef struct {
    int32_t T;                /* tokens, >= 0                                  */
    int32_t H;                /* hidden channels, > 0, multiple of 8 (of 128
                                 for fp8 payloads)                             */
    int32_t E;                /* experts, 1..EP_MAX_EXPERTS                    */
    int32_t k;                /* experts per token, 1..min(E, EP_MAX_TOPK)     */
    int32_t num_partitions;   /* P >= 1, divides E; partition p holds experts
                                 [p*E/P, (p+1)*E/P)                            */
    int32_t mode;             /* ep_layout_mode_t                              */
    int32_t capacity;         /* rows per expert, >= 1 in capacity mode        */
} ep_shape_t;

/* Rows R of the receive buffer for this shape; -1 if the shape is invalid. */
EP_API int64_t ep_recv_rows(const ep_shape_t *shape);

/* Bytes of device workspace ep_get_layout needs for this shape (may be 0);
 * (size_t)-1 if the shape is invalid. */
EP_API size_t ep_layout_workspace_bytes(const ep_shape_t *shape);

/*
 * ep_get_layout -- turn top-k routing into the per-expert layout.
 *
 * Passages: the per-expert token count and the division of experts into
 * partitions (expert e on partition e / (E/P)) follow the low-latency
 * dispatch excerpt quoted in "Redundant atomics in internode_ll" (DeepEP
 * issue #282, question); the order inside an expert follows "Reasons for not
 * calling NVSHMEM public APIs?" (DeepEP issue #18, answer on low-latency
 * mode: the data of one expert keeps its order).  The pages do not give the
 * layout as a separate call; on one GPU the count exchange they describe
 * becomes this call.
 *
 * In:  topk_idx   i32 [T, k]  expert of copy (t, j); -1 = masked slot.
 * Out: counts       i32 [E]    copies routed to each expert (true demand,
 *                              also in capacity mode).
 *      offsets      i32 [E+1]  exclusive prefix sum of counts.
 *      part_counts  i32 [P]    counts summed over each partition.
 *      part_offsets i32 [P+1]  exclusive prefix sum of part_counts.
 *      slot_of      i32 [T, k] receive row of copy (t, j); -1 if masked or
 *                              dropped for capacity.
 *      src_token    i32 [R]    token of each receive row; -1 if the row holds
 *                              no copy.
 *      src_k        i32 [R]    top-k position j of each receive row; -1 if
 *                              the row holds no copy.
 * Order: rows of one expert hold its copies in increasing (t, j), so the
 * result is deterministic and equals a stable sort of the flattened ids.
 *   packed:   slot = offsets[e] + rank(t, j),
 *   capacity: slot = e*capacity + rank if rank < capacity, else dropped
 *             (EP_ERRF_CAPACITY),
 * rank(t, j) = number of copies (t', j') < (t, j) routed to the same expert.
 * workspace: device buffer of ep_layout_workspace_bytes(shape) bytes, owned
 * by the caller, contents on entry ignored; NULL allowed when that is 0.
 * err_flags: EP_ERRF_BAD_EXPERT, EP_ERRF_CAPACITY.
 */
EP_API ep_status_t ep_get_layout(const ep_shape_t *shape, const int32_t *topk_idx,
                          int32_t *counts, int32_t *offsets,
                          int32_t *part_counts, int32_t *part_offsets,
                          int32_t *slot_of, int32_t *src_token, int32_t *src_k,
                          void *workspace, size_t workspace_bytes,
                          uint32_t *err_flags, ep_stream_t stream);

/*
 * ep_get_layout_static -- ep_get_layout without a caller-supplied workspace.
 * The pages have no counterpart of this entry point: it exists for callers
 * that cannot allocate device memory where they compute the layout (code
 * confined to a fixed memory budget owned by a host framework, or a latency-
 * critical path on which a device allocation could stall the device).
 *
 * Same arguments, outputs, ordering and err_flags as ep_get_layout, minus
 * workspace / workspace_bytes.  Scratch comes from a 1 MiB array built into
 * the library (every GPU that loads the library holds it until the process
 * exits): shapes needing more than 1 MiB of layout workspace, i.e.
 * ceil(T*k / 1024) * E * 4 bytes > 1 MiB (about 2^20 routing entries at
 * E = 256), return EP_ERR_UNSUPPORTED; smaller shapes that need no workspace
 * use none.  The array's device address is looked up on the first call that
 * needs it in each device context, with that context current, and reused
 * while the same context lives (a context created later, e.g. after
 * cudaDeviceReset, gets its own lookup); make that first call before any
 * stream capture.  All calls share the array and it keeps the
 * last call's contents (each call writes every entry it reads, so nothing
 * needs clearing); calls whose work overlaps on the GPU race on it and must
 * be ordered by the caller.  Allocates nothing.
 */
EP_API ep_status_t ep_get_layout_static(const ep_shape_t *shape, const int32_t *topk_idx,
                          int32_t *counts, int32_t *offsets,
                          int32_t *part_counts, int32_t *part_offsets,
                          int32_t *slot_of, int32_t *src_token, int32_t *src_k,
                          uint32_t *err_flags, ep_stream_t stream);

/*
 * ep_dispatch -- copy every token's hidden row to each receive row it is
 * routed to (slot_of from ep_get_layout; R = ep_recv_rows(shape)).
 *
 * In:  x        bf16 [T, H], 16-byte aligned.
 *      topk_w   f32 [T, k] routing weights, or NULL.
 *      slot_of  i32 [T, k] receive row of each copy, -1 = none; each
 *               non-negative value should appear at most once (rows written
 *               twice end up with either copy); values outside [-1, R) are
 *               skipped and flagged EP_ERRF_BAD_SLOT.
 * Out: recv     EP_PAYLOAD_BF16:     bf16 [R, H]: recv[slot_of[t,j]] = x[t].
 *               EP_PAYLOAD_FP8_E4M3: e4m3 [R, H]; per token t and channel
 *               block b of 128: s = max(amax, 1e-4) / 448 (fp32, round to
 *               nearest), q = e4m3(x / s) (fp32 division rounded to nearest,
 *               then nearest e4m3, ties to even, saturating at +-448).
 *               16-byte aligned.
 *               EP_PAYLOAD_FP8_E4M3_UE8M0: as E4M3 but s is the smallest
 *               power of two >= max(amax, 1e-4) / 448 (that quotient rounded
 *               to nearest in fp32), so x / s is exact ("Support UE8M0 data
 *               format", referenced from "Redundant atomics in
 *               internode_ll").
 *      recv_scales (fp8 only, else ignored): E4M3: f32 [R, H/128], s of each
 *               block, 16-byte aligned; E4M3_UE8M0: u8 [R, H/128], the biased
 *               exponent e of each block's s = 2^(e - 127).
 *      recv_w   f32 [R] or NULL: recv_w[slot_of[t,j]] = topk_w[t,j]
 *               (needs topk_w).
 * Rows of recv / recv_scales / recv_w that receive no copy are not written.
 * err_flags: EP_ERRF_TIMEOUT, EP_ERRF_BAD_SLOT.
 */
EP_API ep_status_t ep_dispatch(const ep_shape_t *shape, const void *x,
                        const float *topk_w, const int32_t *slot_of,
                        int32_t payload, void *recv, void *recv_scales,
                        float *recv_w, uint32_t *err_flags, ep_stream_t stream);

/*
 * ep_layout_dispatch -- ep_get_layout followed by ep_dispatch, in one launch
 * when the batch is small (T*k <= 2048 and T <= 2048), otherwise as those two
 * calls.  Small decode batches are where a launch matters ("Why does DeepEP
 * LL kernel use double send/recv/signal buffers?", last answer: the design
 * targets high tokens per second), and the v1 low-latency path avoided a
 * separate count exchange ("Why did DeepEP v2 drop the double-buffer
 * design...", question).
 *
 * Arguments, outputs, ordering, checks and err_flags are exactly those of
 * ep_get_layout (topk_idx .. src_k, workspace, workspace_bytes) and
 * ep_dispatch (x, topk_w, payload, recv, recv_scales, recv_w) on the same
 * shape; every output is bit-identical to the two separate calls.  The
 * workspace is only used on the two-call path (size from
 * ep_layout_workspace_bytes).
 */
EP_API ep_status_t ep_layout_dispatch(const ep_shape_t *shape, const int32_t *topk_idx,
                          const void *x, const float *topk_w, int32_t payload,
                          int32_t *counts, int32_t *offsets,
                          int32_t *part_counts, int32_t *part_offsets,
                          int32_t *slot_of, int32_t *src_token, int32_t *src_k,
                          void *recv, void *recv_scales, float *recv_w,
                          void *workspace, size_t workspace_bytes,
                          uint32_t *err_flags, ep_stream_t stream);

/*
 * ep_combine -- weighted top-k reduce of expert outputs back to token order.
 *
 * Passage: combine is the reverse of dispatch and is measured beside it in
 * "Pipeline direct NVLink dispatch with triple-buffered prefetch" (DeepEP PR
 * #693), Validation table (combine GB/s unchanged by the dispatch pipeline,
 * balanced and unbalanced); the pages do not spell out its arithmetic, which
 * is read here as the weighted sum of the token's k expert outputs.
 *
 * In:  y        bf16 [R, H] expert outputs in the receive layout, 16-byte
 *               aligned.
 *      topk_w   f32 [T, k], or NULL for an unweighted sum (weights applied on
 *               the expert side, e.g. from ep_dispatch's recv_w).
 *      slot_of  i32 [T, k] from ep_get_layout (-1 = skipped; values outside
 *               [-1, R) are skipped and flagged EP_ERRF_BAD_SLOT).
 * Out: out      bf16 [T, H], 16-byte aligned:
 *               out[t] = bf16( sum_{j: slot_of[t,j] >= 0} topk_w[t,j] * y[slot_of[t,j]] ),
 *               accumulated in fp32 in increasing j from 0 (each product and
 *               sum rounded to nearest), rounded once to bf16 (nearest even).
 *               A token with no valid slot gets 0.
 * err_flags: EP_ERRF_BAD_SLOT.
 */
EP_API ep_status_t ep_combine(const ep_shape_t *shape, const void *y,
                       const float *topk_w, const int32_t *slot_of, void *out,
                       uint32_t *err_flags, ep_stream_t stream);

/*
 * ep_combine_fp8 -- ep_combine over fp8 expert outputs (the e4m3 variant of
 * the combine the pages measure beside dispatch, "Pipeline direct NVLink
 * dispatch with triple-buffered prefetch", Validation table).
 *
 * In:  y        e4m3 [R, H] expert outputs in the receive layout, 16-byte
 *               aligned; H % 128 == 0.
 *      y_scales payload EP_PAYLOAD_FP8_E4M3: f32 [R, H/128] (4-byte aligned);
 *               EP_PAYLOAD_FP8_E4M3_UE8M0: u8 [R, H/128] biased exponents,
 *               scale = 2^(e - 127).
 *      topk_w, slot_of, out, err_flags as ep_combine.
 * Each element is dequantised as v = value(code) * scale (fp32 product,
 * rounded to nearest), then out[t] = bf16( sum_j topk_w[t,j] * v ) in fp32 in
 * increasing j, as ep_combine.
 */
EP_API ep_status_t ep_combine_fp8(const ep_shape_t *shape, const void *y,
                       const void *y_scales, int32_t payload,
                       const float *topk_w, const int32_t *slot_of, void *out,
                       uint32_t *err_flags, ep_stream_t stream);

/*
 * ep_combine_src -- the combine addressed from the expert side.  The caller
 * holds, for every row of the expert-major buffer, the token and top-k
 * position the row was dispatched from (ep_get_layout's src_token / src_k)
 * and, optionally, the row's own weight (ep_dispatch's recv_w: the routing
 * information that travels with each token, "Pipeline direct NVLink dispatch
 * with triple-buffered prefetch", Summary), instead of the token-side slot_of.
 * Copy j of token t is the row r with (src_token[r], src_k[r]) = (t, j); the
 * rows are read in place (no copy of y is made).
 *
 * In:  y, y_scales, payload  as ep_combine (payload EP_PAYLOAD_BF16, y_scales
 *               NULL) or ep_combine_fp8 (the two fp8 payloads).
 *      row_w    f32 [R] weight of each row, or NULL for an unweighted sum.
 *      src_token, src_k  i32 [R]: the pair each row holds, src_token = -1 in a
 *               row that holds no copy.  Each pair appears in at most one row
 *               (as ep_get_layout writes them; if several rows claim a pair,
 *               which one is used is unspecified).  A row whose pair lies
 *               outside [0,T) x [0,k) (other than src_token = -1) is skipped
 *               and flags EP_ERRF_BAD_SLOT.
 *      workspace  device memory of ep_combine_src_workspace_bytes(shape)
 *               bytes, 4-byte aligned, caller-owned; its contents on entry do
 *               not matter.  It receives the token-side map rebuilt from the
 *               source maps, [T, k] rows then [T, k] weights.
 * Out: out      bf16 [T, H]: exactly what ep_combine / ep_combine_fp8 give
 *               with slot_of[t,j] = r and topk_w[t,j] = row_w[r] (bit for
 *               bit): fp32 sum in increasing j, one rounding to bf16; a pair
 *               that no row holds (a dropped or masked copy) adds nothing.
 * err_flags: EP_ERRF_BAD_SLOT.
 */
EP_API size_t ep_combine_src_workspace_bytes(const ep_shape_t *shape);
EP_API ep_status_t ep_combine_src(const ep_shape_t *shape, const void *y,
                       const void *y_scales, int32_t payload, const float *row_w,
                       const int32_t *src_token, const int32_t *src_k, void *out,
                       void *workspace, size_t workspace_bytes,
                       uint32_t *err_flags, ep_stream_t stream);

/* Static description of a status code. */
EP_API const char *ep_status_string(ep_status_t status);

/* The same function under the shorter name of the original interface plan. */
EP_API const char *ep_status_str(ep_status_t status);

/* Detail of the last non-EP_OK status returned on the calling thread
 * ("" if none).  The pointer stays valid until the next call on this thread. */
EP_API const char *ep_last_error(void);

/* ABI version of this library (major * 100 + minor). */
EP_API int32_t ep_abi_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* EP_GB300_H_ */
