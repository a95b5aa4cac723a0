/*
 * fa.h — C ABI of the exact, IO-aware attention forward for GB300 (sm_103a).
 *
 * Operation (per batch b, query head h, query row i):
 *     S_ij   = scale * <Q[b,h,i,:], K[b,g,j,:]>,   g = h / (Hq / Hkv)
 *     O[b,h,i,:] = sum_j softmax_j(S_i.) * V[b,g,j,:]      over visible j
 *     LSE[b,h,i] = ln sum_j exp(S_ij)                       over visible j
 * with "visible" = every key when causal == 0, and key j <= query i when
 * causal != 0 (top-left alignment, for any Nq, Nkv).
 *
 * Where it is defined:
 *   - "flash attention v3 paper" search page (cidian.kuaisou.com), first
 *     snippet: standard attention S = QK^T, P = row-softmax(S), O = PV
 *     (scale and mask omitted there);
 *   - "Hacker News Digest — gpu-computing" (hckr.top), section "Алгоритм
 *     Flash Attention 2": scale = DIM**-0.5 multiplies Q K^T, the loop over
 *     (batch, query tile) and over key/value tiles with an in-place online
 *     softmax; section "v1 — базовая версия", item 3: the running max and
 *     denominator recurrence;
 *   - "Flash Attention (Kutarisa Kwemheni)" (aiunderstanding.org), summary
 *     and FAQ: the result is exact attention, computed tile by tile so the
 *     N x N score matrix never reaches HBM.
 * GQA head sharing and the LSE output are this library's specification; the
 * pages do not define them.
 *
 * All functions are thread-safe and callable from any host thread.
 *
 * Device memory.  The library's own device memory is the status word read by
 * fa_last_device_error and the fixed array behind fa_fwd_noalloc, both part
 * of the loaded module.  One stated exception: fa_fwd, fa_fwd_qk8 and
 * fa_fwd_host take the scratch some shapes need (split-KV partials, the
 * stream schedule's partials and flags; fa_fwd_workspace_size gives the
 * size) from a per-device stream-ordered pool, and that pool keeps up to
 * 64 MiB of freed scratch reserved between calls so a later call does not
 * map memory again (on a 152-SM GB300 no shape needs more than about 30 MB;
 * anything above 64 MiB returns to the device at the next synchronisation).
 * Callers that want no such reserve use fa_fwd_ws (their own scratch) or
 * fa_fwd_noalloc (the fixed array).
 *
 * Set-up.  The first call into the library on a device (any entry point
 * that touches the device) checks the compute capability, sets the kernels'
 * shared-memory limits, creates the pool and looks up the device addresses
 * of the module's arrays, once per device with that device current; make
 * that first call before any stream capture on the device.
 *
 * TMA tensor maps are encoded on the host and cached per (pointer, extents,
 * box, element type) in a 64-entry table: repeated calls on the same
 * buffers encode nothing (fa_tensor_map_encodes counts the encodings).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_VALUE = 1, /* null pointer, dimension < 1, Hq % Hkv != 0,
                                 non-finite scale, size beyond the limits   */
    FA_ERR_UNSUPPORTED = 2,   /* D not in {64, 128, 192, 256}, or the
                                 current device is not compute capability
                                 10.3 (sm_103)                              */
    FA_ERR_MISALIGNED = 3,    /* q, k, v or o not 16-byte aligned, or lse not
                                 4-byte aligned (TMA needs 16 bytes)        */
    FA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (launch,
                                 device query, tensor-map encoding)         */
    FA_ERR_TIMEOUT = 5        /* a kernel's bounded wait ran out (reported by
                                 fa_last_device_error after a sync)         */
} fa_status;

/*
 * fa_fwd — attention forward on bf16 tensors, fp32 log-sum-exp.
 *
 *   q    device pointer, bf16 [B, Hq,  Nq,  D], contiguous (row-major)
 *   k    device pointer, bf16 [B, Hkv, Nkv, D], contiguous
 *   v    device pointer, bf16 [B, Hkv, Nkv, D], contiguous
 *   o    device pointer, bf16 [B, Hq,  Nq,  D], contiguous; written
 *   lse  device pointer, fp32 [B, Hq,  Nq], contiguous; written; may be NULL
 *   B, Hq, Hkv, Nq, Nkv, D   sizes; Hq must be a multiple of Hkv (query head
 *        h reads kv head h / (Hq / Hkv)); D in {64, 128, 192, 256}
 *        (192 and 256, and causal shapes at 64, run a kernel with one
 *        128-row query tile per CTA)
 *   scale  finite fp32 multiplier of Q K^T (typically 1/sqrt(D))
 *   causal 0: every key visible; nonzero: key j visible to query i iff j <= i
 *   stream a cudaStream_t (as void*); NULL means the legacy default stream
 *
 * Ownership: the caller owns every buffer; nothing is retained after the
 * call returns.  o and lse must not overlap q, k, v or each other.
 *
 * Behaviour: arguments are validated on the host and an error is returned
 * before anything is launched; on FA_OK the work is enqueued on `stream`
 * and the call returns without synchronising.  Faults during execution
 * surface at the next synchronisation of that stream; a bounded wait that
 * ran out is reported by fa_last_device_error().  O is rounded to bf16
 * (round-to-nearest-even); arithmetic is fp32 with bf16 tensor-core inputs.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int Hq, int Hkv, int Nq, int Nkv, int D,
           float scale, int causal, void* stream);

/*
 * fa_fwd_ws — fa_fwd with caller-provided scratch memory.
 *
 * When the 256-row query blocks of a call fill fewer than half the SMs
 * (decode-like or small-batch shapes), each block's key/value range is cut
 * into contiguous pieces processed by separate CTAs ("split-KV", the
 * FlashDecoding-style partition named on the "flash attention v3 paper"
 * search page, second snippet).  Each piece leaves fp32 partial results
 * (unnormalised O, running max, running sum per row) in scratch memory and
 * a merge kernel combines them with the same rescaling the online softmax
 * uses between key/value tiles.  The stream schedule (see fa_fwd_schedule)
 * also needs scratch: one fp32 partial slot and eight flags per CTA.
 * fa_fwd takes that scratch from a per-device stream-ordered pool;
 * fa_fwd_ws uses `workspace` instead.
 *
 *   workspace        device pointer, 16-byte aligned, at least
 *                    fa_fwd_workspace_size() bytes; may be NULL when that
 *                    size is 0.  Its contents on entry do not matter; the
 *                    call overwrites it.  Calls that may run concurrently
 *                    must not share it.
 *   workspace_bytes  its size in bytes
 * Other arguments, ownership and errors as fa_fwd; FA_ERR_INVALID_VALUE if
 * the workspace is missing or too small, FA_ERR_MISALIGNED if unaligned.
 */
int fa_fwd_ws(const void* q, const void* k, const void* v, void* o,
              float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
              float scale, int causal, void* workspace,
              size_t workspace_bytes, void* stream);

/*
 * fa_fwd_workspace_size — bytes of scratch fa_fwd_ws needs for this shape on
 * the current device; 0 when the shape is not split (then no scratch is
 * used).  Writes *bytes and returns FA_OK; argument errors as fa_fwd.
 */
int fa_fwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                          int causal, size_t* bytes);

/*
 * fa_fwd_qk8 — fa_fwd with Q and K in 8-bit floating point (e4m3).
 *
 * The low-precision MMA path that "Flash Attention на 5090 в CUDA C++" sets
 * as its goal (introduction; "Что дальше": MXFP8/NVFP4 MMA), in its plainest
 * form: S = Q K^T runs on the tensor cores as an e4m3 x e4m3 product with
 * fp32 accumulation (tcgen05 kind::f8f6f4), with one descale factor per
 * tensor; P V stays bf16.  Block-scaled formats are not supported.
 *
 *   q8   device pointer, e4m3 (1 byte) [B, Hq,  Nq,  D], contiguous
 *   k8   device pointer, e4m3 (1 byte) [B, Hkv, Nkv, D], contiguous
 *   v, o, lse, B, Hq, Hkv, Nq, Nkv, causal, stream: as for fa_fwd
 *   D    must be 128 (FA_ERR_UNSUPPORTED otherwise)
 *   scale, q_descale, k_descale   the scores are
 *        scale * q_descale * k_descale * (q8 . k8), with q8 and k8 taken
 *        exactly as e4m3 values; the descales must be finite and > 0
 *        (FA_ERR_INVALID_VALUE otherwise)
 *
 * Ownership, validation, asynchrony, split-KV scratch and error behaviour
 * are those of fa_fwd.
 */
int fa_fwd_qk8(const void* q8, const void* k8, const void* v, void* o,
               float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
               float scale, float q_descale, float k_descale, int causal,
               void* stream);

/*
 * fa_fwd_mxfp8 — fa_fwd with Q and K in MXFP8: 8-bit floating point (e4m3)
 * with one power-of-two scale per 32 consecutive head-dim elements of a row.
 *
 * The block-scaled low-precision MMA that "Flash Attention на 5090 в CUDA
 * C++" sets as its goal (introduction; "Что дальше": MXFP8/NVFP4 MMA), in
 * its 8-bit form: S = Q K^T runs on the tensor cores as a block-scaled
 * e4m3 x e4m3 product (tcgen05 kind::mxf8f6f4, one scale per 32 elements of
 * each operand) with fp32 accumulation; P V stays bf16.  The scores are
 *     S[i][j] = scale * sum_b 2^(qs[i][b] - 127) 2^(ks[j][b] - 127)
 *                       * sum_{d = 32b .. 32b+31} q8[i][d] k8[j][d],
 * the dot products of the exactly dequantised rows.
 *
 *   q8       device pointer, e4m3 (1 byte) [B, Hq,  Nq,  D], contiguous
 *   k8       device pointer, e4m3 (1 byte) [B, Hkv, Nkv, D], contiguous
 *   v, o, lse, B, Hq, Hkv, Nq, Nkv, scale, causal, stream: as for fa_fwd
 *   q_scale  device pointer, ue8m0 bytes [B, Hq,  Nq,  D / 32], contiguous,
 *            4-byte aligned: qs above (value 2^(byte - 127))
 *   k_scale  device pointer, ue8m0 bytes [B, Hkv, Nkv, D / 32], likewise
 *   D        must be 128 (FA_ERR_UNSUPPORTED otherwise)
 *
 * Runs one 128-row query tile per CTA (the scale factors live in tensor
 * memory beside S and O), with no split-KV.  Ownership, validation,
 * asynchrony and errors as fa_fwd; FA_ERR_INVALID_VALUE for a NULL scale
 * pointer, FA_ERR_MISALIGNED for one not 4-byte aligned.
 */
int fa_fwd_mxfp8(const void* q8, const void* k8, const void* v,
                 const void* q_scale, const void* k_scale, void* o,
                 float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                 float scale, int causal, void* stream);

/* Schedules reported by fa_fwd_schedule (and forced by fa_set_schedule). */
enum {
    FA_SCHEDULE_AUTO = -1,    /* fa_set_schedule only: choose per shape    */
    FA_SCHEDULE_PLAIN = 0,    /* one CTA per unit of query rows            */
    FA_SCHEDULE_SPLIT_KV = 1, /* key/value ranges split over CTAs, merged
                                 by a second kernel (see fa_fwd_ws)        */
    FA_SCHEDULE_STREAM = 2,   /* equal share of all work per CTA           */
    FA_SCHEDULE_PERSIST = 3   /* one CTA per SM over a list of whole units */
};

/*
 * fa_fwd_schedule — how fa_fwd, fa_fwd_ws, fa_fwd_qk8 and fa_fwd_noalloc run
 * this shape on the current device (the choice depends only on the shape
 * and the device's SM count, for any nonzero scale: a call whose scale is 0
 * runs FA_SCHEDULE_PLAIN where this reports FA_SCHEDULE_PERSIST).
 *
 *   *kind            FA_SCHEDULE_PLAIN: one CTA per unit of query rows (a
 *                    pair of 128-row tiles; one tile for D 192/256 and for
 *                    causal D 64), each over all its keys;
 *                    FA_SCHEDULE_SPLIT_KV: each unit's key/value blocks cut
 *                    into *pieces ranges, one CTA each, then a merge kernel;
 *                    FA_SCHEDULE_STREAM (no causal mask, D 64 or 128): the
 *                    (tile pair, key/value block) items of the whole call
 *                    dealt out in equal contiguous runs of *blocks_per_cta,
 *                    one per CTA, when whole pairs would leave SMs idle in
 *                    their last wave.  A pair cut between CTAs is finished
 *                    by the CTA holding its last block, which combines the
 *                    others' fp32 partials in its epilogue (no second
 *                    kernel).  The grid is a cooperative launch (all
 *                    CTAs resident at once, at most one per SM), so every
 *                    CTA a merger waits for is running; where the device
 *                    cannot hold the whole grid at once (e.g. an SM limit
 *                    set for the process) the launch fails and the call
 *                    returns FA_ERR_CUDA.  A wait that runs out reports
 *                    FA_ERR_TIMEOUT through fa_last_device_error.
 *                    FA_SCHEDULE_PERSIST (causal mask, D 64 or 128, bf16
 *                    Q/K, no split, K and V of the call within 96 MiB,
 *                    fewer than 2^31 pairs of query tiles):
 *                    at most one CTA per SM, each walking a list of whole
 *                    pairs of 128-row query tiles, longest first and dealt
 *                    out in a snake order, so short causal pairs share a
 *                    CTA's set-up and one pair's epilogue overlaps the next
 *                    pair's first products.
 *   *ctas            CTAs of the attention kernel
 *   *pieces          key/value ranges per unit (split-KV), else 1
 *   *blocks_per_cta  128-key blocks per CTA (stream), else 0
 * Non-causal grouped-query shapes are counted as they run: the Hq / Hkv
 * query heads of a group form one head of (Hq / Hkv) * Nq rows.  Argument
 * errors as fa_fwd_workspace_size; all four outputs must be non-NULL.
 */
int fa_fwd_schedule(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                    int causal, int* kind, int* ctas, int* pieces,
                    int* blocks_per_cta);

/*
 * fa_fwd_schedule_for — fa_fwd_schedule for a GPU with `sms` SMs, without
 * touching any device (the choice depends only on the shape, the SM count
 * and fa_set_schedule); also writes the scratch fa_fwd_ws would need there
 * to *workspace.  FA_ERR_INVALID_VALUE for sms < 1 or a NULL output;
 * other argument errors as fa_fwd_workspace_size.
 */
int fa_fwd_schedule_for(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                        int causal, int sms, int* kind, int* ctas,
                        int* pieces, int* blocks_per_cta,
                        size_t* workspace);

/*
 * fa_set_schedule — force the schedule of later calls, process-wide, for
 * testing and tuning (the default, FA_SCHEDULE_AUTO, chooses per shape from
 * an estimate of each schedule's time).
 *
 *   FA_SCHEDULE_PLAIN   one CTA per unit of query rows; also no split-KV
 *                       and no persistent schedule
 *   FA_SCHEDULE_STREAM  the stream schedule wherever it exists (no causal
 *                       mask, D 64 or 128), with any share per CTA, so a
 *                       pair may be cut into many pieces; other shapes keep
 *                       the automatic choice
 *   FA_SCHEDULE_AUTO    back to the automatic choice
 *
 * Returns FA_ERR_INVALID_VALUE for any other value.  The setting is one
 * atomic word read when a call plans its launch (and by
 * fa_fwd_workspace_size and fa_fwd_schedule): a workspace sized under one
 * setting may be too small under another.  Results agree with the oracle
 * under every setting; only the time and the scratch size change.
 */
int fa_set_schedule(int kind);

/*
 * fa_fwd_host — fa_fwd on host buffers: copies Q, K, V in, runs the forward,
 * copies O and LSE out, overlapping the copies with the computation.
 *
 * The pages describe no such call; host-resident inputs are where a caller
 * without device-side producers starts, and the host link is slower than
 * the forward (on GB300 about 200 GB/s each way: 42 MB of bf16 Q, K, V for
 * the 4096 x 8192 x 8-head shape take 0.2 ms, twice the forward).  The call
 * splits the job into at most 4 chunks of consecutive (batch, kv head)
 * groups, each a forward of its own (a group's rows are contiguous in the
 * [B, H, N, D] layout): chunk c's K, V and Q are copied in on a side stream,
 * its forward runs on `stream` (its small size lets the split-KV schedule
 * spread it over the GPU), and its O and LSE are copied out on a second side
 * stream while later chunks copy in and compute.
 *
 *   q_host, k_host, v_host  host pointers, layouts as fa_fwd's q, k, v; page-
 *                           locked (cudaHostAlloc / cudaHostRegister) for the
 *                           copies to be asynchronous and overlap
 *   o_host, lse_host        host pointers receiving O and LSE; lse_host may
 *                           be NULL exactly when lse_dev is NULL
 *   q_dev .. lse_dev        device buffers of the full sizes, as fa_fwd's
 *                           arguments (16-byte aligned; lse 4-byte aligned)
 *   B .. causal             as fa_fwd
 *   stream                  the work is ordered after the caller's earlier
 *                           work on `stream`, and `stream` completes only
 *                           after the last copy out: synchronise it before
 *                           reading o_host
 * Errors as fa_fwd; FA_ERR_INVALID_VALUE for a NULL host pointer (checked
 * before anything is enqueued).  If an error occurs after the first copy was
 * enqueued, `stream` is still made to wait for every copy already enqueued,
 * so synchronising it is enough before the buffers are reused; the outputs
 * are then incomplete.  Calls from different host threads on one device are
 * serialised while they enqueue (they share the side streams); their GPU
 * work may still overlap.
 */
int fa_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                void* o_host, float* lse_host, void* q_dev, void* k_dev,
                void* v_dev, void* o_dev, float* lse_dev, int B, int Hq,
                int Hkv, int Nq, int Nkv, int D, float scale, int causal,
                void* stream);

/* Size of the fixed scratch array behind fa_fwd_noalloc (32 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * fa_fwd_noalloc — fa_fwd for callers that must not allocate device memory.
 *
 * The pages describe no such call; it exists for callers that cannot call
 * cudaMalloc or take memory from an allocator while they run: for example
 * code that reserves all device memory up front and forbids allocation
 * afterwards (a serving process with a fixed memory plan, a plugin inside a
 * host framework that owns the allocator), or code on a latency-critical
 * path where an allocation's cost or failure is not acceptable.
 *
 * It computes exactly what fa_fwd computes, with the same arguments, and
 * allocates nothing: the split-KV scratch some shapes need (see fa_fwd_ws)
 * lives in one fixed device array of FA_NOALLOC_SCRATCH_BYTES bytes that is
 * part of the library and stays resident on every device that has loaded
 * it until the process exits.  Shapes that need more scratch than that
 * (fa_fwd_workspace_size() > FA_NOALLOC_SCRATCH_BYTES) are rejected with
 * FA_ERR_INVALID_VALUE before anything is launched.  The scratch a shape
 * needs grows with the GPU's SM count, not with the sequence lengths; on a
 * 152-SM GB300 every supported shape needs at most about 30 MB, so none is
 * rejected there.
 *
 * The array's device address is looked up once per device, with that
 * device current, by the first call into the library on that device (see
 * "Set-up" above); make that first call before any stream capture.  All
 * calls on a device share the one array: two calls
 * whose kernels may overlap on the GPU (different streams, no ordering
 * between them) race on it and can corrupt each other's results.  Calls
 * ordered on one stream are safe.  Each call overwrites every part of the
 * array that it later reads, so nothing needs clearing between calls.
 */
int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                   float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                   float scale, int causal, void* stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* fa_status_string(int status);

/*
 * fa_last_device_error — FA_OK, or FA_ERR_TIMEOUT if any kernel of this
 * library on the current device gave up a bounded wait since the previous
 * query.  Reads and clears a device-side word (synchronising copy); call it
 * after synchronising the streams the kernels ran on.  Returns FA_ERR_CUDA
 * if the word cannot be read.
 */
int fa_last_device_error(void);

/*
 * fa_probe_bounded_wait — enqueue a one-warp kernel on `stream` that waits
 * on a shared-memory barrier nothing will ever complete, with a limit of
 * `timeout_ns` nanoseconds (1 .. 10^9), then records FA_ERR_TIMEOUT in the
 * device word read by fa_last_device_error() and returns.  It exercises the
 * same bounded-wait routine the attention kernel uses, so a caller can check
 * that an expired wait ends in an error status instead of a hang.
 * Returns FA_ERR_INVALID_VALUE for a limit outside the range.
 */
int fa_probe_bounded_wait(long long timeout_ns, void* stream);

/*
 * fa_probe_flag_wait — as fa_probe_bounded_wait, for the other bounded wait
 * the kernels use: a one-warp kernel waits (acquire loads) for a global
 * 64-bit flag to reach a value nothing will ever publish — the wait a stream-
 * schedule CTA makes for another CTA's partial — with a limit of
 * `timeout_ns` (1 .. 10^9), then records FA_ERR_TIMEOUT for
 * fa_last_device_error() and returns.  FA_ERR_INVALID_VALUE for a limit
 * outside the range.
 */
int fa_probe_flag_wait(long long timeout_ns, void* stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int fa_version(void);

/*
 * fa_tensor_map_encodes — how many TMA tensor maps the library has encoded
 * (cuTensorMapEncodeTiled calls) since it was loaded, over all threads and
 * devices.  A call whose four maps (Q, K, V, O) are in the cache adds
 * nothing.  For tests and tuning; touches no device.
 */
size_t fa_tensor_map_encodes(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
