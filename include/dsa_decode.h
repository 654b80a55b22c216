/*
 * dsa_decode.h -- C ABI of the GB300 sparse-attention decode path.
 *
 * One decode step of one unit (a (session, layer) pair) runs five steps:
 * DSA indexer scoring + Top-K, hot-cache gather, Q8G64 dequantisation,
 * absorbed-MLA attention over the selected rows, and append with batched
 * write-back. Every call below is batched over U units in one launch
 * sequence, enqueues asynchronously on the caller's CUDA stream, and returns
 * after host-side argument checks.
 *
 * Sources (page titles; section headings in the original and in English):
 *   [P3]  "从总共 1M 到 15+ 路 × 1M：GLM-5.3 KV Cache 换出的容量突破"
 *         (From 1M total to 15+ x 1M: GLM-5.3 KV-cache offload)
 *   [ALG] "算法层：从注意力、KV Cache 到 FFN 与 MoE"
 *         (Algorithm layer: from attention and KV cache to FFN and MoE)
 *   [QNT] "量化不是压缩包：从模型分层到 4-bit 推理的工程真相"
 *         (Quantization is not a zip file)
 *
 * Conventions
 *   - The caller owns all memory. "device" pointers are CUDA device memory
 *     (or a device-accessible alias of pinned host memory where stated).
 *     No call allocates memory; scratch is a caller-provided workspace whose
 *     size the matching *_workspace() query returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Return value: DSA_OK (0) or a negative DSA_ERR_* code. A host-side
 *     error enqueues nothing. DSA_ERR_CUDA means a launch failed.
 *   - Errors found on the device (an index out of bounds, an append beyond
 *     capacity, a query value outside the attention kernel's range) are OR-ed
 *     into the caller's device word `dev_err` as DSA_DEVERR_* bits; the kernel
 *     skips the offending access and carries on. Read the word back after the
 *     stream completes and pass it to dsa_check().
 *   - bf16 and fp16 values are passed as their 16-bit patterns.
 */
#ifndef DSA_DECODE_H
#define DSA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- constants */

#define DSA_OK 0
#define DSA_ERR_ARG (-1)          /* null pointer or out-of-range argument        */
#define DSA_ERR_SHAPE (-2)        /* unsupported shape (e.g. K > 4096, bad H)     */
#define DSA_ERR_WS (-3)           /* workspace missing or too small               */
#define DSA_ERR_CUDA (-4)         /* a CUDA runtime call or launch failed         */
#define DSA_ERR_DEVICE_CHECK (-6) /* dsa_check(): the device word is non-zero     */
#define DSA_ERR_SCRATCH_LIMIT (-7) /* problem larger than a fixed built-in scratch */

#define DSA_DEVERR_BOUNDS 0x1     /* a position/slot index was out of range       */
#define DSA_DEVERR_CAPACITY 0x2   /* append beyond the unit's lmax                */
#define DSA_DEVERR_QRANGE 0x4     /* attention operand outside the fp16 range    */
#define DSA_DEVERR_TIMEOUT 0x8    /* a bounded wait inside a kernel gave up        */
#define DSA_DEVERR_ROUND 0x10     /* hot_gather round below the unit's last round */
#define DSA_DEVERR_STATE 0x20     /* export/restore of a unit not flushed / not matching */

#define DSA_ROW_BYTES 656         /* Q8G64 MLA row: 512 int8 + 8 fp16 + 64 bf16   */
#define DSA_LAT_DIM 512
#define DSA_ROPE_DIM 64
#define DSA_IDX_HEADS 8
#define DSA_IDX_DIM 64
#define DSA_RING_ROWS 64
#define DSA_MAX_K 4096
#define DSA_MAX_ROWS 8            /* query rows per unit per step (MTP verify)   */
#define DSA_MAX_ATTN_K 2048       /* selected rows per attention query row       */
#define DSA_ROUND_AUTO (-1)       /* hot_gather: use the unit's gather-call count */

#define DSA_CLS_HOT 0             /* read from an HBM hot slot                    */
#define DSA_CLS_RING 1            /* read from the GPU recent ring                */
#define DSA_CLS_RAM 2             /* read from the host RAM mirror                */
#define DSA_CLS_PAD 3             /* no position (-1 in topk_idx)                 */

#define DSA_WARM_EMPTY 0
#define DSA_WARM_LAST_S 1

#define DSA_POLICY_RING 0         /* ring replacement skipping pinned slots      */
#define DSA_POLICY_CLOCK 1        /* clock with reference bits (needs `ref`)    */

/* state[] word indices of a unit (int64 each) */
#define DSA_ST_LEN 0              /* logical rows (history length)               */
#define DSA_ST_RAM 1              /* positions < this are in the RAM mirror       */
#define DSA_ST_HAND 2             /* ring-replacement hand                        */
#define DSA_ST_EPOCH 3            /* gather-call counter (pins are per call)      */
#define DSA_ST_WRITEBACKS 4       /* number of write-back batches issued          */
#define DSA_ST_ROUND 5            /* last hot_gather round + 1 (0: none yet)      */
#define DSA_ST_WORDS 8

/*
 * One unit's cache state. An array of these lives in DEVICE memory and is
 * passed to the calls as `units`. All pointers are device-accessible; the
 * struct itself is written only by the caller (the kernels update the arrays
 * it points to).
 *
 *   keys       bf16 [lmax][64]   indexer keys; position p at keys + 64*p.
 *   slots      u8   [S][656]     hot-cache rows (HBM).
 *   slot_pos   i32  [S]          position held by each slot, -1 = empty.
 *   pos_slot   i32  [lmax]       slot holding each position, -1 = none.
 *   fill_round i32  [S]          round of the slot's last fill (-1 = warm).
 *   pin_epoch  i32  [S]          internal: gather call that last pinned it.
 *   ring       u8   [64][656]    recent ring; position p at row p % 64.
 *   mirror     u8   [lmax][656]  RAM mirror: device alias of pinned host
 *                                memory from dsa_host_alloc() (offloaded), or
 *                                HBM (the fully resident variant).
 *   state      i64  [8]          DSA_ST_* words.
 *   slots_n    S (>= 1).
 *   policy     DSA_POLICY_RING or DSA_POLICY_CLOCK (see hot_gather).
 *   lmax       capacity in positions (history + all appends).
 *   ref        u8   [S]          reference bits (clock policy; may be NULL
 *                                for the ring policy).
 * 16-byte alignment is required for keys, slots, ring and mirror: a unit
 * that breaks it is skipped by every kernel and sets DSA_DEVERR_BOUNDS.
 */
typedef struct dsa_unit {
  uint16_t* keys;
  uint8_t* slots;
  int32_t* slot_pos;
  int32_t* pos_slot;
  int32_t* fill_round;
  int32_t* pin_epoch;
  uint8_t* ring;
  uint8_t* mirror;
  int64_t* state;
  int32_t slots_n;
  int32_t policy;
  int64_t lmax;
  uint8_t* ref;
} dsa_unit;

/* ------------------------------------------------------------ housekeeping */

/* ABI version of this header (returns 2). */
int dsa_abi_version(void);

/* Static text for a DSA_* status code. */
const char* dsa_status_string(int status);

/* Map a device error word read back from `dev_err` to a status:
 * DSA_OK if it is 0, else DSA_ERR_DEVICE_CHECK. */
int dsa_check(int32_t dev_err_value);

/*
 * Diagnostic of the failure path that every kernel's bounded waits share: a
 * one-CTA kernel waits on a barrier phase for at most `limit_cycles` SM
 * cycles. With `complete` = 0 nothing completes the phase, the wait gives up
 * and DSA_DEVERR_TIMEOUT is OR-ed into *dev_err (so dsa_check reports
 * DSA_ERR_DEVICE_CHECK) while the context stays usable; with `complete` != 0
 * the phase completes first and the word is untouched. Nothing is left in
 * flight either way.
 */
int dsa_wait_selftest(int64_t limit_cycles, int32_t complete, int32_t* dev_err, void* stream);

/*
 * Pinned, mapped host memory for a unit's RAM mirror ([P3] section
 * "第三次决策：让 GPU 直接管理热缓存" (third decision: the GPU manages the hot
 * cache): a miss reads the *registered* RAM mirror directly; section
 * "GPU 管缓存也会犯错": registration is done ahead of time so no first-use
 * registration stall lands on the decode path).
 *   host_ptr  out: host address (page-locked, mapped, portable).
 *   dev_ptr   out: the device-accessible alias to put in dsa_unit.mirror.
 * (cudaHostAlloc, mapped and portable.)
 * Returns DSA_ERR_CUDA if the allocation fails. Free with dsa_host_free().
 * This is setup, not part of a decode step.
 */
int dsa_host_alloc(void** host_ptr, void** dev_ptr, size_t bytes);
int dsa_host_free(void* host_ptr);

/*
 * Initialise U units' cache state for histories of l0[u] rows that are
 * already in the mirror (positions [0, l0) are RAM-resident, the ring is
 * empty, hand = 0).
 *   units    device dsa_unit[U].
 *   l0       device int64 [U]; 0 <= l0[u] <= lmax.
 *   warm     DSA_WARM_EMPTY: every slot empty. DSA_WARM_LAST_S: slot i holds
 *            position l0 - n + i for n = min(S, l0), fill_round -1, and its
 *            bytes are copied from the mirror. Reference bits (when `ref` is
 *            set) start set for the occupied slots and clear for the others.
 *   max_slots, max_lmax  host bounds: max over units of S and of lmax
 *            (they size the grid).
 * Also clears pin_epoch and the DSA_ST_* words. A unit whose l0 is outside
 * [0, lmax] or whose S < 1 is left untouched and sets DSA_DEVERR_BOUNDS.
 * Finally it reads one word of every host page of each mirror ([0, lmax)
 * rows), so that the GPU's address translations for the whole mirror exist
 * before decoding: misses read random rows spread over the mirror, and
 * without this the first decode steps pay for the translations (about 3 ms
 * per step on a 20 GiB mirror in 32 units, fading over ~20 steps).
 */
int hc_init(const dsa_unit* units, int32_t U, int32_t warm, const int64_t* l0,
            int32_t max_slots, int64_t max_lmax, int32_t* dev_err, void* stream);

/*
 * The last part of hc_init alone: one read of every host page of each unit's
 * mirror ([0, lmax) rows), enqueued on `stream`. The address translations it
 * sets up serve kernels of the same context: measured on a GB300, gathers on
 * an SM partition's streams (dsa_partition_split, a green context) paid for
 * them again over their first 25 to 80 decode steps (up to 5 ms per step)
 * although hc_init had run on an ordinary stream. Call it once on a stream of
 * each partition whose kernels read the mirrors. Units whose arrays are not
 * 16-byte aligned are skipped. max_lmax: host bound, max over units of lmax.
 */
int dsa_touch_mirror(const dsa_unit* units, int32_t U, int64_t max_lmax, void* stream);

/* --------------------------------------------- A1 + A2: DSA score and Top-K */

/*
 * [P3] section "起点：把容量和当前计算的工作集分开" (starting point): the DSA
 * indexer selects the Top-2048 history positions that MLA attention then
 * consumes; section "第一次决策" (first decision): this stays the exact GPU
 * path with a BF16 query.
 *
 * For each unit u and query row r, over the positions s in [0, L) with
 * L = state[DSA_ST_LEN] at the start of the call:
 *     I[r][s] = sum_h w[r][h] * max(0, sum_d q[r][h][d] * keys[s][d])
 * (8 indexer heads, d = 64, float32 accumulation), and keeps the K largest
 * scores, equal scores going to the lower position. Output: the K selected
 * positions in ascending order, padded with -1 when L < K.
 *
 *   units     device dsa_unit[U] (keys and state[DSA_ST_LEN] are read).
 *   q         device bf16 [U][R][8][64].
 *   w         device float [U][R][8].
 *   topk_idx  device int32 [U][R][K] (written).
 *   max_len   host bound: max over units of L (sizes the grid).
 *   ws        device workspace of dsa_score_topk_workspace(U, R, max_len)
 *             bytes, 16-byte aligned. It must be zero-filled once before its
 *             first use; every call leaves it ready for the next.
 *   q         must be 16-byte aligned as well (read as 16-byte vectors).
 * Shapes: 1 <= U, 1 <= R <= 8, 1 <= K <= 4096.
 */
size_t dsa_score_topk_workspace(int32_t U, int32_t R, int64_t max_len);
int dsa_score_topk(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
                   const uint16_t* q, const float* w, int32_t* topk_idx,
                   int64_t max_len, void* ws, size_t ws_bytes,
                   int32_t* dev_err, void* stream);

/*
 * The two halves of dsa_score_topk, for callers that run them on different
 * streams (dsa_score_topk is dsa_score then dsa_topk_select on one stream).
 * Same arguments and workspace; the workspace of one call pair must not be
 * used by another call until dsa_topk_select has run.
 *   dsa_score        scores the units into the workspace (ordered score keys,
 *                    histograms, group maxima): one launch of the persistent
 *                    score kernel, whose grid fills the SMs that `stream` may
 *                    use (the SMs of the partition it belongs to, see
 *                    dsa_partition_split, else the whole device).
 *   dsa_topk_select  selects the Top-K from what dsa_score left in the
 *                    workspace and clears it for the next call; it must be
 *                    ordered after dsa_score (same stream, or an event).
 */
int dsa_score(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
              const uint16_t* q, const float* w, int64_t max_len,
              void* ws, size_t ws_bytes, int32_t* dev_err, void* stream);
int dsa_topk_select(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
                    int32_t* topk_idx, int64_t max_len, void* ws,
                    size_t ws_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------- SM partitions (schedule) */

/*
 * Partitions of the current device's SMs (CUDA green contexts): kernels
 * launched on a partition's streams run only on its SMs. Their use: the
 * indexer's score kernel streams every key from HBM on a persistent grid that
 * holds all the SMs it may use until it ends, so the rest of another batch's
 * step (selection, slot assignment, gather, attention) can run beside it only
 * on SMs it was not given. Kernels of this library size their grids to the
 * partition of the stream they are launched on.
 *
 * dsa_partition_split splits the device in two. The device's SMs come as
 * co-scheduling groups (SMs of one GPU processing cluster, 8 on a GB300)
 * plus some SMs that form no whole group. `first` takes those leftovers,
 * then whole groups until it holds at least min_sms; `second` takes the
 * groups left, whole, so that thread-block clusters (the Top-K select
 * launches 8-CTA clusters) fit there.
 *   min_sms  1 <= min_sms < the device's SM count.
 *   first    out (may be NULL: not created): the first partition.
 *   second   out (may be NULL: not created): the second partition.
 * Returns DSA_ERR_ARG for a count that leaves nothing for a requested second
 * partition, DSA_ERR_CUDA where the driver has no green contexts or refuses.
 * The caller owns the partitions (dsa_partition_destroy).
 *
 * dsa_partition_sms     the SMs of a partition.
 * dsa_partition_stream  a new non-blocking stream of the partition (a
 *                       cudaStream_t, owned by the partition, valid until
 *                       dsa_partition_destroy).
 * dsa_stream_wait_stream  work queued later on `waiter` waits for the work
 *                       queued so far on `signaller`. Either may be a
 *                       partition's stream or an ordinary stream of the
 *                       device: an event recorded on a partition's stream
 *                       must come from its own context, so ordinary events
 *                       (cudaEventRecord) cannot order partition streams;
 *                       this call can.
 * dsa_partition_destroy waits for the work queued on the partition's streams,
 *                       then releases them and the green context.
 * A partition is used from one host thread at a time; its streams are not
 * captured into CUDA graphs.
 */
typedef struct dsa_partition dsa_partition;
int dsa_partition_split(int32_t min_sms, dsa_partition** first, dsa_partition** second);
int dsa_partition_sms(const dsa_partition* part);
int dsa_partition_stream(dsa_partition* part, void** stream);
int dsa_stream_wait_stream(void* waiter, void* signaller);
int dsa_partition_destroy(dsa_partition* part);

/*
 * dsa_score_topk without a caller workspace, for callers that cannot
 * allocate device memory: for example code that runs inside a host framework
 * which owns every device allocation and forbids cudaMalloc, or a loop that
 * must never stall on the allocator. The pages have no counterpart to this
 * entry point; it computes exactly what dsa_score_topk computes (same
 * arguments minus ws/ws_bytes) and enqueues the same kernels.
 *
 * Its scratch is one array of 5.375 MiB compiled into this library (device
 * memory that every GPU which loads the library keeps until the process
 * exits). Limits: U * R <= 16 and max_len <= 65,536; larger problems return
 * DSA_ERR_SCRATCH_LIMIT and enqueue nothing.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (the device must be current). Make that first call
 *     before capturing any stream into a CUDA graph.
 *   - Every call shares the one array: calls that may overlap on the GPU (two
 *     streams, or two host threads) race and give wrong results. Calls in one
 *     stream are ordered and safe.
 *   - Each call clears the histogram part of the array (a cudaMemsetAsync on
 *     `stream`) before scoring; no call allocates or frees memory.
 */
int dsa_score_topk_noalloc(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
                           const uint16_t* q, const float* w, int32_t* topk_idx,
                           int64_t max_len, int32_t* dev_err, void* stream);

/*
 * Selection reuse across layers ([P3] section "起点": some later layers reuse
 * the selection, while every layer keeps its own KV). Score only the source
 * units (dsa_score_topk on a units array holding just them, output src_topk),
 * then fill every unit's selection: rows of unit u of topk_idx <- rows of
 * unit src_of[u] of src_topk. A unit reuses another's selection when its
 * src_of points at that unit's scored rows; src_of outside [0, Us) sets
 * DSA_DEVERR_BOUNDS and leaves the unit unchanged. A source should share the
 * consumer's history (same session).
 *   topk_idx device int32 [U][R][K] (written); src_topk device int32 [Us][R][K];
 *   src_of   device int32 [U].
 */
int dsa_reuse_selection(int32_t* topk_idx, const int32_t* src_topk, int32_t U, int32_t Us, int32_t R,
                        int32_t K, const int32_t* src_of, int32_t* dev_err, void* stream);

/* -------------------------------------------------------- A3: hot gather */

/*
 * [P3] section "第三次决策：让 GPU 直接管理热缓存" (third decision): the GPU
 * looks up the hot slot of every selected position; a hit reads VRAM, a miss
 * reads the registered RAM mirror, forming the compact selected set.
 * [P3] section "GPU 管缓存也会犯错：跨 block 可见性与置换长扫描" (cross-block
 * visibility and long replacement sweeps): slots filled in round r are hits
 * only from round r + 1; duplicate misses of a round read RAM; slots in use
 * this round are pinned; rows not yet written back are served by the recent
 * ring; replacement is a ring that skips pinned slots.
 *
 * Per unit, with the state as it is when the call starts:
 *   RING if p >= state[DSA_ST_RAM]; else HOT if pos_slot[p] = s >= 0 and
 *   fill_round[s] < round; else RAM. HOT slots are pinned for this call.
 *   The distinct RAM positions that hold no slot, in ascending order, take
 *   the eligible slots (not pinned, fill_round < round) in cyclic order from
 *   the hand: the old position loses its mapping, the slot gets the new
 *   position, fill_round = round and the mirror row's bytes; then
 *   hand = last slot + 1 (mod S). Misses beyond the eligible slots are served
 *   from RAM and not inserted.
 *
 *   topk_idx  device int32 [U][R][K] (ascending per row, -1 padded).
 *   cls       device u8 [U][R][K]: DSA_CLS_* per entry (written).
 *   rows      device u8 [U][R][K][656]: the compact selected rows, bytes
 *             exactly as read from their source (PAD entries are zeroed).
 *   counters  device int32 [U][4]: HOT, RING, RAM entries, slots filled.
 *   ws        device workspace of hot_gather_workspace(U, R, K) bytes.
 * With DSA_POLICY_CLOCK (the policy the pages replaced; [P3] section "GPU 管缓存
 * 也会犯错": with a full window, every reference bit set and 1% misses, the few
 * missing blocks swept far), each slot has a reference bit: a HOT hit sets
 * it; the victims are found by the clock hand's walk from `hand`, which
 * passes over pinned slots, slots filled in this round and slots already
 * taken, clears a set bit and passes on, and takes a slot whose bit is
 * clear; after two turns it stops. A fill sets the bit; hand = last victim +
 * 1. (Computed with two block scans over the cyclic order, not a serial walk:
 * the eligible slots with a clear bit come first, then those with a set
 * bit; the bits the first turn passes are cleared.)
 * Shapes: 1 <= U, 1 <= R <= 8, 1 <= K <= 4096. `round` must not decrease
 * from call to call on a unit (a repeated round is allowed): a call whose
 * round is below the unit's previous one would break the visibility rule, so
 * it sets DSA_DEVERR_ROUND and leaves that unit's state unchanged (its
 * entries come back DSA_CLS_PAD with zeroed rows and zero counters). A negative
 * `round` (DSA_ROUND_AUTO) uses each unit's state[DSA_ST_EPOCH], the number of
 * earlier hot_gather calls on it, so one call per decode step gives rounds
 * 0, 1, 2, ... with fixed arguments (e.g. inside a captured CUDA graph).
 */
size_t hot_gather_workspace(int32_t U, int32_t R, int32_t K);
int hot_gather(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
               int32_t round, const int32_t* topk_idx, uint8_t* cls,
               uint8_t* rows, int32_t* counters, void* ws, size_t ws_bytes,
               int32_t* dev_err, void* stream);

/*
 * The two halves of hot_gather, for callers that overlap them with other work:
 * hot_gather_assign classifies, pins and assigns victims and updates the
 * cache state (cls, counters, the workspace's fill list); hot_gather_copy
 * then writes the compact rows (and the inserted misses' slot bytes) from
 * that workspace. hot_gather = hot_gather_assign + hot_gather_copy on one
 * stream. Ordering:
 *   - the copy must follow its assign (same units, topk_idx, cls, ws), and must
 *     finish before the next hot_gather_assign on the same units starts (that
 *     assign may evict slots this copy reads; a HOT row whose slot mapping
 *     changed under the copy is zeroed and sets DSA_DEVERR_BOUNDS);
 *   - after the assign, kv_append_writeback with A = 1 may run concurrently
 *     with the copy: it writes the ring row of position LEN - 64 (below RAM,
 *     never RING in this round), the key of position LEN and mirror rows at
 *     or above RAM (read from the ring in this round), none of which the copy
 *     reads; the next step's dsa_score_topk (into another topk buffer) may then
 *     overlap the copy and the attention as well.
 */
int hot_gather_assign(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t round,
                      const int32_t* topk_idx, uint8_t* cls, int32_t* counters, void* ws, size_t ws_bytes,
                      int32_t* dev_err, void* stream);
int hot_gather_copy(const dsa_unit* units, int32_t U, int32_t R, int32_t K, const int32_t* topk_idx,
                    const uint8_t* cls, uint8_t* rows, void* ws, size_t ws_bytes, int32_t* dev_err,
                    void* stream);

/* ---------------------------------- A4 + A5: dequant and MLA decode attention */

/*
 * [ALG] section "2. Attention": softmax(Q K^T / sqrt(d_k)) V; section
 * "3. KV Cache": MLA keeps the normalised latent and the RoPE part, INT8 per
 * group for the latent. [QNT] section "三、基本思路": w_hat = scale * q with
 * one scale per group (G64: 64 latent values). [P3] section "起点": a row is
 * 512 B latent + 16 B scales + 128 B RoPE = 656 B.
 *
 * Absorbed MLA over the compact rows, for each unit u, query row r, head h:
 *   c_j[d]  = int8_j[d] * fp16scale_j[d / 64]           (d < 512)
 *   logit_j = scale * (q_lat[h] . c_j + q_rope[h] . rope_j)
 *   out[h]  = sum_j softmax_j(logit) * c_j,   lse[h] = log sum_j exp(logit_j)
 * over the entries j with topk_idx >= 0; with none, out = 0 and lse = -inf.
 *
 *   q_lat   device bf16 [U][R][H][512];  q_rope device bf16 [U][R][H][64].
 *           The tensor-core operands are fp16 with fp32 accumulation: |q| and
 *           |int8 * scale| must stay below 65504, else DSA_DEVERR_QRANGE is
 *           set. Each operand is rounded once to fp16 (relative error <= 2^-11).
 *   rows    device u8 [U][R][K][656] (hot_gather's output), 16-byte aligned;
 *           the workspace too (both are read with bulk copies; otherwise
 *           DSA_ERR_ARG).
 *   topk_idx device int32 [U][R][K] (only the sign is used: -1 = padding).
 *   out     device float [U][R][H][512];  lse device float [U][R][H] or NULL.
 *   ws      device workspace of mla_decode_attn_workspace(U, R, H, K) bytes:
 *           per (unit, query row) and run of selected rows (at most 16), one
 *           64 x 512 fp32 partial output and its 64 row maxima and sums,
 *           written by the first kernel of the call and read by the second
 *           (in L2).
 * Shapes: H in {16, 32, 48, 64}, 1 <= K <= DSA_MAX_ATTN_K, U * R <= 65535.
 * Two kernels: per (unit, query row) the selected rows are cut into chunks
 * of 64 and the chunks into runs, one CTA per run (as many runs as fill the
 * GPU once), each an online-softmax part over its rows; then a merge of the
 * parts (one block per (unit, query row) and 32 output columns).
 */
size_t mla_decode_attn_workspace(int32_t U, int32_t R, int32_t H, int32_t K);
int mla_decode_attn(int32_t U, int32_t R, int32_t H, int32_t K,
                    const uint16_t* q_lat, const uint16_t* q_rope,
                    const uint8_t* rows, const int32_t* topk_idx, float scale,
                    float* out, float* lse, void* ws, size_t ws_bytes,
                    int32_t* dev_err, void* stream);

/*
 * hot_gather followed by mla_decode_attn in one call, without the compact
 * rows: the attention kernel reads each selected row straight from its
 * source (HOT slot, ring, RAM mirror) as this call's classification found it,
 * and writes each inserted miss's row to its victim slot ([P3] section
 * "第三次决策": hits read VRAM, misses read the registered RAM mirror, and
 * attention consumes the gathered set). Classification, pins, visibility,
 * replacement, counters, cache state and out/lse are exactly those of
 * hot_gather + mla_decode_attn; only the compact `rows` buffer is not
 * produced. Duplicate misses of different query rows each read the mirror.
 * Each row is staged by one 656-byte bulk copy from its source, the next
 * chunk's rows while the current chunk is multiplied; the attention's runs
 * fill the SMs of the stream's partition (or the device).
 *   Arguments as in hot_gather and mla_decode_attn; ws holds
 *   hot_gather_attn_workspace(U, R, H, K) bytes, 256-byte aligned.
 *   Shapes: those of mla_decode_attn.
 * Ordering: the step's kv_append_writeback must not run concurrently with
 * this call (the call reads ring rows that an append of several rows may
 * overwrite).
 */
size_t hot_gather_attn_workspace(int32_t U, int32_t R, int32_t H, int32_t K);
int hot_gather_attn(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t H, int32_t round,
                    const int32_t* topk_idx, const uint16_t* q_lat, const uint16_t* q_rope, float scale,
                    uint8_t* cls, int32_t* counters, float* out, float* lse, void* ws, size_t ws_bytes,
                    int32_t* dev_err, void* stream);

/* ------------------------------------------- A6: append and batched write-back */

/*
 * [P3] section "第三次决策": new KV goes to a GPU recent ring and is written
 * back to the RAM history in batches; section "第二次决策" (second decision):
 * 64-row batches replaced per-row, per-layer transfers; small logs are copied
 * by compute kernels rather than DMA operations.
 *
 * For each unit and a = 0..A-1, with p = state[DSA_ST_LEN]:
 *   ring[p % 64] = new_rows[a]; keys[p] = new_keys[a]; LEN += 1;
 *   when LEN - state[DSA_ST_RAM] == 64, the 64 ring rows of positions
 *   [RAM, RAM + 64) are stored to mirror (41,984 B, by the kernel) and
 *   RAM += 64.
 * An append with p >= lmax sets DSA_DEVERR_CAPACITY and is dropped.
 *   new_rows device u8 [U][A][656];  new_keys device bf16 [U][A][64].
 * Shapes: 1 <= U, 1 <= A <= 64.
 * Ordering: it must follow the step's hot_gather (which reads LEN and RAM),
 * and may run concurrently with the step's mla_decode_attn (on another
 * stream): it writes only the ring row and key of position LEN and mirror
 * rows >= RAM, none of which this step's gathered rows came from.
 */
int kv_append_writeback(const dsa_unit* units, int32_t U, int32_t A,
                        const uint8_t* new_rows, const uint16_t* new_keys,
                        int32_t* dev_err, void* stream);

/*
 * kv_append_writeback for new rows given in bf16: each row is Q8G64-quantised
 * once on the GPU before it enters the ring ([P3] section "第二次决策": the
 * owner quantises a new KV row once and moves the 656-byte packed row; [QNT]
 * section "三、基本思路": symmetric q = round(w / scale), one scale per 64
 * values). Per group of 64 latent values: scale = fp16_rn(max|w| / 127) and
 * q = clamp(rint(w / scale), -127, 127), both divisions IEEE fp32; a group
 * whose scale is 0 or not finite in fp16 gets scale 0 and zero codes. The
 * RoPE part is stored as given. Everything else as kv_append_writeback.
 *   new_latent device bf16 [U][A][512]; new_rope device bf16 [U][A][64];
 *   new_keys device bf16 [U][A][64].
 */
int kv_append_quantize(const dsa_unit* units, int32_t U, int32_t A, const uint16_t* new_latent,
                       const uint16_t* new_rope, const uint16_t* new_keys, int32_t* dev_err,
                       void* stream);

/*
 * [P3] section "容量优化必须通过会话生命周期" (capacity work must survive the
 * session lifecycle): before exporting or restoring the full history, flush
 * the log, wait for write-back, and check that the RAM row count has reached
 * the logical row count.
 *
 * Stores the partial batch [RAM, LEN) from the ring to the mirror and sets
 * RAM = LEN. After the stream completes, the mirror holds every row.
 */
int kv_flush(const dsa_unit* units, int32_t U, int32_t* dev_err, void* stream);

/* ------------------------------------------------- session export and restore */

/*
 * [P3] section "容量优化必须通过会话生命周期" (capacity work must survive the
 * session lifecycle): a session is saved and restored, and before exporting
 * or restoring the full history the log is flushed, the write-back waited
 * for, and the RAM row count checked against the logical row count.
 *
 * A unit's snapshot holds its DSA_ST_* words, slot map (slot_pos,
 * fill_round), reference bits, recent ring and indexer keys [0, LEN); the
 * RAM mirror is the caller's own host memory and is not copied. Its size is
 * dsa_snapshot_bytes(S, lmax); unit u's snapshot is at snap + u * snap_stride
 * (snap_stride >= the size for the largest S and lmax, a multiple of 16;
 * snap 16-byte aligned; device memory or a mapped host alias from
 * dsa_host_alloc).
 *
 * dsa_export: call after kv_flush on the same stream. A unit whose RAM row
 * count is not its logical row count (not flushed) is not exported and sets
 * DSA_DEVERR_STATE.
 * dsa_restore: into units with the same S and lmax >= LEN whose mirrors hold
 * the exported history rows [0, LEN). Restores the words, slot map, bits,
 * ring and keys, rebuilds pos_slot, clears the pins and re-reads every slot's
 * bytes from the mirror. A unit whose S differs, whose lmax is too small or
 * whose snapshot was not flushed is left as it is and sets DSA_DEVERR_STATE.
 * max_slots, max_lmax: host bounds over the units (they size the grids).
 */
size_t dsa_snapshot_bytes(int32_t S, int64_t lmax);
int dsa_export(const dsa_unit* units, int32_t U, uint8_t* snap, size_t snap_stride, int32_t max_slots,
               int64_t max_lmax, int32_t* dev_err, void* stream);
int dsa_restore(const dsa_unit* units, int32_t U, const uint8_t* snap, size_t snap_stride, int32_t max_slots,
                int64_t max_lmax, int32_t* dev_err, void* stream);

/*
 * [P3] section "容量优化必须通过会话生命周期": a large append (prefill of many
 * new rows) first restores the full history of GPU MLA KV from RAM, appends,
 * and decode then returns to the hot cache.
 *
 * Copies each unit's history [0, LEN) as dense 656-byte rows into
 * dst + u * dst_rows * 656: rows below RAM from the mirror (over the host
 * link), the rest from the recent ring. Rows at or past dst_rows are not
 * copied. dst: device memory, 16-byte aligned, U * dst_rows * 656 bytes.
 */
int kv_restore_full(const dsa_unit* units, int32_t U, uint8_t* dst, int64_t dst_rows, int32_t* dev_err,
                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_DECODE_H */
