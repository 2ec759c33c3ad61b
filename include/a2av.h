/*
 * a2av.h -- C ABI of a GB300 (sm_103a) variable-size all-to-all with
 * device-resident splits (all_to_all_vdev).
 *
 * The operation ("[a2av] Improve tuning for 4 GPUs", pytorch PR 154580,
 * section "Problem": nvshmem_all_to_all_vdev, each rank sending a
 * variable-size chunk to every peer, with the split sizes held on the device):
 *
 *   W ranks, r, p in [0, W).  S[r][p] = in_splits[r*W + p] rows go from rank
 *   r to peer p.  Rank r's input holds its chunks back to back in peer order,
 *   starting at row 0; peer p's output receives them back to back in
 *   source-rank order, starting at row 0:
 *
 *     out[p] rows [out_off[p][r], out_off[p][r] + S[r][p])
 *        = in[r] rows [in_off[r][p], in_off[r][p] + S[r][p])
 *     in_off[r][p]  = sum_{q<p} S[r][q]      out_off[p][r] = sum_{q<r} S[q][p]
 *
 *   and out_splits_offsets[p][0][r] = S[r][p], out_splits_offsets[p][1][r] =
 *   out_off[p][r].  A row is row_bytes bytes, copied bit for bit.
 *
 * Here the W ranks are W pairs of buffers in the HBM of ONE GPU; the exchange
 * is one kernel launch that reads the split matrix on the device (no host
 * round trip), scans it, writes out_splits_offsets and moves every chunk.
 * The pages' NVSHMEM design split its CTAs between the peers and, when the
 * peers are few, the data-parallel dimension within each chunk (same page,
 * section "Change"); this library balances bytes, not chunks, across CTAs.
 *
 * Conventions for every entry point:
 *  - Return value: A2AV_OK or a negative a2av_status_t.  Host-detectable
 *    errors are returned synchronously and launch nothing.
 *  - Device pointers are CUDA device (or managed) addresses on the device
 *    that was current when the handle was created; that device must be
 *    current on every call.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  The caller owns every buffer and the stream; the library never
 *    allocates, frees or retains them.
 *  - Not thread-safe per handle: one host thread at a time per handle.
 */
#ifndef A2AV_H_
#define A2AV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest number of ranks one exchange supports. */
#define A2AV_MAX_RANKS 32

typedef enum {
  A2AV_OK = 0,
  A2AV_ERR_INVALID_ARG = -1, /* a host-checked argument is wrong */
  A2AV_ERR_UNSUPPORTED = -2, /* a valid request this build does not serve (W > 32) */
  A2AV_ERR_CUDA = -3,        /* a CUDA runtime call failed (no device, launch failure...) */
  A2AV_ERR_BAD_SPLITS = -4,  /* device-detected: the split matrix is invalid */
  A2AV_ERR_TIMEOUT = -5,     /* device-detected: a bounded wait inside a kernel gave up */
  A2AV_ERR_BAD_INDEX = -6    /* device-detected: a dispatch key or source row, or a combine
                                position, is out of range */
} a2av_status_t;

/* Copy engine selection (a2av_set_path). */
typedef enum {
  A2AV_PATH_AUTO = 0,   /* bulk when every row and buffer is 16-byte aligned, else staged */
  A2AV_PATH_VECTOR = 1, /* 16-byte register loads/stores, realigned by warp shuffles */
  A2AV_PATH_BULK = 2,   /* cp.async.bulk global->shared->global (aligned exchanges only) */
  A2AV_PATH_STAGED = 3  /* cp.async.bulk granules -> shared -> realigned 16-byte stores */
} a2av_path_t;

typedef struct a2av_handle a2av_handle;

/*
 * a2av_create -- make a handle for exchanges among `world_size` ranks on the
 * current CUDA device.
 *
 *  world_size          W, 1 <= W <= A2AV_MAX_RANKS (W > 32: A2AV_ERR_UNSUPPORTED).
 *  in_capacity_rows    rows every input buffer can hold; sum_p S[r][p] above it is
 *                      rejected on the device.  0 = unchecked.
 *  out_capacity_rows   rows every output buffer can hold; sum_r S[r][p] above it is
 *                      rejected on the device.  0 = unchecked.
 *  out                 receives the handle (host pointer, must not be NULL).
 *
 * Allocates a small device status word (cudaMalloc) on the current device.
 * Reads five environment variables once: A2AV_PATH (an a2av_path_t number,
 * the initial engine), A2AV_CTAS_PER_SM (the initial grid override), A2AV_PDL
 * (0 turns programmatic dependent launch off; see a2av_run),
 * A2AV_DISPATCH_ORDER (which batches a2av_dispatch orders in its one-launch
 * order kernel: 0 none, 1 -- the default -- rows under 64 bytes, 2 every
 * row size, 3 also the batches its one-CTA-per-rank count takes) and
 * A2AV_DEBUG_STARVE -- a test hook: 1 makes the first CTA of every bulk or
 * staged launch (and the first warp of the fused dispatch's and combine's
 * bulk gather) arm its first stage for 16 more bytes than its copies
 * deliver, so that stage never completes; 2 makes the grid barrier of the
 * one-launch dispatch and combine kernels wait for one CTA more than the
 * grid holds.  Either way the bounded wait gives up after about a second and
 * the run records A2AV_ERR_TIMEOUT.  No copy is left in flight, nothing is
 * written past the failed wait, and the context stays usable.  Never set it
 * outside tests.
 * Errors: A2AV_ERR_INVALID_ARG (W < 1, negative capacity, out == NULL),
 * A2AV_ERR_UNSUPPORTED, A2AV_ERR_CUDA (no usable device).
 */
int a2av_create(int world_size, int64_t in_capacity_rows, int64_t out_capacity_rows,
                a2av_handle **out);

/*
 * a2av_run -- one all_to_all_vdev over the handle's W ranks, enqueued on
 * `stream` as a single kernel launch; returns without waiting for it.  The
 * launch uses programmatic stream serialization (unless A2AV_PDL=0): its
 * CTAs may be scheduled while the previous kernel on `stream` still runs,
 * and wait on the device for that kernel to finish, its writes visible,
 * before they read or write anything -- stream order is kept, only the
 * launch latency is hidden.
 *
 *  in_ptrs            HOST array of W device pointers: rank r's input, its chunks
 *                     back to back in peer order from row 0.  Read only.  A NULL
 *                     entry is a rank with no input (it must send 0 rows).
 *  in_splits_dev      DEVICE int64 [W][W], row-major by source rank: S[r][p] at
 *                     in_splits_dev[r*W + p].  Read only; 8-byte aligned.
 *  out_ptrs           HOST array of W device pointers: peer p's output.  Written
 *                     only in its first sum_r S[r][p] rows.  A NULL entry is a
 *                     peer that receives nothing (it must receive 0 rows).
 *  out_splits_offsets_dev  DEVICE int64 [W][2][W]: written with
 *                     [p][0][r] = S[r][p] and [p][1][r] = out_off[p][r] (rows).
 *  row_bytes          bytes per row, >= 1, any value (no alignment needed).
 *  stream             cudaStream_t as void*.
 *
 * Memory rules: no output may overlap an input, the split matrix or another
 * output; inputs may share memory.  Input and output buffers may also be
 * host memory that the device can address (pinned or registered memory, or
 * system memory reached over NVLink-C2C: zero-copy over the host link).  The
 * library looks at every buffer pointer (cudaPointerGetAttributes) and runs
 * the vector engine, whose plain loads and stores reach any of them, unless
 * every buffer is device memory; the bulk and staged engines' cp.async.bulk
 * copies are applied to device memory only, whatever path was requested.
 * The answer for the handle's last two sets of buffer pointers is
 * remembered; a2av_set_path and a2av_set_grid clear that memory (call one
 * after freeing a buffer and allocating memory of another kind at the same
 * address).  Bytes of an input past its last chunk are
 * never used and bytes of an output past its last received row are never
 * written.  (Whole 16-byte-aligned granules that hold a needed input byte may
 * be loaded and their other bytes discarded; such loads never leave the
 * granule and so never fault.)
 *
 * Split validity, checked on the device before anything is written:
 * S[r][p] >= 0; S[r][p] <= 2^62 / (W * row_bytes); sum_p S[r][p] <=
 * in_capacity_rows and sum_r S[r][p] <= out_capacity_rows when those are
 * nonzero; 0 rows for a NULL buffer.  Invalid splits write NOTHING (no output
 * byte, no out_splits_offsets entry) and record A2AV_ERR_BAD_SPLITS in the
 * handle's status word, read by a2av_status.
 *
 * Streams: a small exchange on a side stream beside long kernels that hold
 * every SM (GEMMs) gets SMs only between those kernels unless its stream has
 * a higher priority.  Measured on one GB300 (a 10 MB keyed-jagged exchange,
 * about 16 us alone, beside 8192^3 bf16 GEMMs on the default-priority main
 * stream): 254 us per step on a default-priority side stream, 25 us on a
 * stream created with the highest priority
 * (cudaStreamCreateWithPriority), at no cost to the GEMMs.  Give
 * latency-sensitive exchanges a high-priority stream.
 *
 * Host errors (nothing launched): A2AV_ERR_INVALID_ARG for a NULL handle or
 * array, a NULL split or out_splits_offsets pointer, a misaligned split
 * pointer, row_bytes < 1, or a current device other than the handle's;
 * A2AV_ERR_CUDA when the launch fails.
 */
int a2av_run(a2av_handle *h, const void *const *in_ptrs, const int64_t *in_splits_dev,
             void *const *out_ptrs, int64_t *out_splits_offsets_dev, int64_t row_bytes,
             void *stream);

/*
 * a2av_combine -- the reverse exchange: every peer sends each chunk it
 * received back to the rank it came from (the return path of an MoE token
 * dispatch).  The pages define only the forward exchange; this is that same
 * exchange applied to the transposed split matrix S', S'[p][r] = S[r][p],
 * which a dispatch's out_splits_offsets already holds (its row 0 for peer p).
 * One kernel launch on `stream`, like a2av_run.
 *
 *  in_ptrs            HOST array of W device pointers: peer p's buffer laid out
 *                     like the dispatch's output (chunks in source-rank order).
 *  dispatch_splits_offsets_dev  DEVICE int64 [W][2][W]: the out_splits_offsets
 *                     a2av_run wrote for the dispatch (only rows [p][0][*] are read).
 *  out_ptrs           HOST array of W device pointers: rank r's buffer receives,
 *                     in peer order, the rows it sent -- the dispatch input's
 *                     layout, so combine(dispatch(x)) == x byte for byte.
 *  out_splits_offsets_dev  DEVICE int64 [W][2][W]: written with
 *                     [r][0][p] = S[r][p] and [r][1][p] = sum_{q<p} S[r][q].
 *  row_bytes, stream  as in a2av_run.
 *
 * Capacities, validity checks, errors and memory rules are a2av_run's, with
 * the combine's own inputs and outputs; dispatch_splits_offsets_dev counts as
 * an input and must not overlap any output.
 */
int a2av_combine(a2av_handle *h, const void *const *in_ptrs,
                 const int64_t *dispatch_splits_offsets_dev, void *const *out_ptrs,
                 int64_t *out_splits_offsets_dev, int64_t row_bytes, void *stream);

/* Largest number of keys (W * keys_per_peer) a fused dispatch sorts by. */
#define A2AV_MAX_DISPATCH_KEYS 1024

/*
 * a2av_dispatch_workspace_bytes -- device workspace a2av_dispatch needs for
 * `world_size` ranks, `keys_per_peer` keys per peer and at most
 * `max_items_per_rank` items on any rank; -1 for arguments a2av_dispatch
 * would reject.  The workspace is caller-owned scratch, 256-byte aligned.
 */
int64_t a2av_dispatch_workspace_bytes(int world_size, int keys_per_peer,
                                      int64_t max_items_per_rank);

/*
 * a2av_dispatch -- fused dispatch preparation: the exchange of a2av_run on
 * rows that are not yet grouped by destination.  The pages take the split
 * matrix as given; this entry point also builds it, the step before the
 * exchange in an MoE dispatch ("MoE related region", PR 154580) or an
 * embedding-key exchange (torchrec PR 2570, "EmbeddingKey alltoall").
 *
 * Rank r has rows_per_rank[r] source rows at rows_ptrs[r] (row_bytes each)
 * and items_per_rank[r] = m_r items.  Item i names a source row
 * src_row_ptrs[r][i] (int32, in [0, rows_per_rank[r])) and a key
 * key_ptrs[r][i] (int32, in [0, W * keys_per_peer)); its destination peer is
 * key / keys_per_peer.  Rank r's items, ordered stably by key (ties by item
 * index), are its virtual input: S[r][p] = the number of items with
 * destination p, and the exchange then proceeds exactly as a2av_run on that
 * virtual input, which is never materialised (rows are gathered straight
 * from rows_ptrs into the outputs).  An MoE top-k dispatch is items
 * (token t, choice k) with src_row = t and key = expert id (keys_per_peer =
 * experts per rank); the peer receives rows ordered by (source rank, local
 * expert, token).
 *
 *  rows_ptrs, rows_per_rank, items_per_rank, src_row_ptrs, key_ptrs:
 *                     HOST arrays of W entries (pointers to device memory for
 *                     the *_ptrs).  Read only.
 *  out_ptrs, out_splits_offsets_dev: as in a2av_run.
 *  sorted_pos_ptrs    HOST array of W device int64 [m_r] arrays: written with
 *                     each item's position in its rank's key order (the
 *                     permutation an MoE combine needs to put rows back).
 *  in_splits_dev      DEVICE int64 [W][W] or NULL: written with S.
 *  workspace          DEVICE scratch of at least
 *                     a2av_dispatch_workspace_bytes(W, keys_per_peer,
 *                     max_r m_r) bytes, 256-byte aligned, not shared with a
 *                     dispatch in flight.
 *
 * Launches on `stream` (a2av_last_dispatch reports which):
 *  - at most 4096 items over all ranks (and W * W * keys_per_peer <= 2048):
 *    ONE kernel, no workspace use, no memset -- every block counts all the
 *    keys itself, derives the split matrix and the plan, then places and
 *    copies its share of the items;
 *  - rows shorter than 64 bytes (see A2AV_DISPATCH_ORDER at a2av_create),
 *    when every item fits the grid's registers (about 1.5 M items over all
 *    ranks on a GB300) and the workspace holds the per-block counts: a
 *    memset of the workspace's first 256 + 8 * W * W bytes, then ONE
 *    cooperative kernel (every block resident at once): each block counts
 *    a chunk of one rank's items, the blocks exchange their counts through
 *    the workspace and one grid barrier (bounded: about a second, then
 *    A2AV_ERR_TIMEOUT), and each block places and copies its chunk;
 *  - otherwise a memset of the workspace's first 256 bytes, then: per-range
 *    key counts and each item's rank within its 256-item range (the scan of
 *    the counts over groups of ranges done by that kernel's last block of
 *    each rank, or, for ranks with very many groups, by a second kernel;
 *    one kernel per rank does both when every rank has at most 2048 items
 *    and W * keys_per_peer <= 256), then the row copy, which alone writes
 *    the caller's buffers: a cp.async.bulk gather for 16-byte aligned rows
 *    above 2 KiB to 32 KiB in device memory, register copies otherwise (for
 *    rows shorter than 64 bytes, one kernel places and copies the rows of
 *    each range after checking the split matrix).
 * Errors: host -- A2AV_ERR_INVALID_ARG (NULL arrays, keys_per_peer < 1,
 * negative counts, a small or misaligned workspace), A2AV_ERR_UNSUPPORTED
 * (W * keys_per_peer > A2AV_MAX_DISPATCH_KEYS, counts above 2^31 - 1);
 * device -- A2AV_ERR_BAD_INDEX for a key or source row out of range,
 * A2AV_ERR_BAD_SPLITS for a capacity or NULL-buffer violation (the handle's
 * output capacity applies; inputs are checked by source-row index) and
 * A2AV_ERR_TIMEOUT when a bounded wait runs out.  On a device-detected
 * BAD_INDEX or BAD_SPLITS nothing is written: no output row, no
 * out_splits_offsets, sorted_pos or in_splits entry.
 */
int a2av_dispatch(a2av_handle *h, int keys_per_peer, const void *const *rows_ptrs,
                  const int64_t *rows_per_rank, const int32_t *const *src_row_ptrs,
                  const int32_t *const *key_ptrs, const int64_t *items_per_rank,
                  void *const *out_ptrs, int64_t *out_splits_offsets_dev,
                  int64_t *const *sorted_pos_ptrs, int64_t *in_splits_dev, int64_t row_bytes,
                  void *workspace, int64_t workspace_bytes, void *stream);

/* Most exchanges a2av_run_multi takes in one launch. */
#define A2AV_MAX_EXCHANGES 4

/* One exchange of an a2av_run_multi call: the arguments of a2av_run. */
typedef struct {
  const void *const *in_ptrs;       /* HOST array of W input pointers */
  const int64_t *in_splits_dev;     /* DEVICE int64 [W][W] */
  void *const *out_ptrs;            /* HOST array of W output pointers */
  int64_t *out_splits_offsets_dev;  /* DEVICE int64 [W][2][W] */
  int64_t row_bytes;
} a2av_exchange_t;

/*
 * a2av_run_multi -- `count` independent exchanges over the handle's W ranks
 * in ONE kernel launch, e.g. the bag lengths and the keys of a keyed-jagged
 * embedding batch (the key all-to-all of "Different nccl stream within
 * EmbeddingKey alltoall", torchrec PR 2570, with the lengths that cut the
 * keys into bags), or MoE tokens and their per-token scales.  Each entry
 * means exactly what the same arguments mean to a2av_run, with its own
 * splits and row size; the result is that of `count` a2av_run calls.  Small
 * exchanges are bound by launch and prologue latency, which the exchanges
 * of one call share.
 *
 *  count      1 <= count <= A2AV_MAX_EXCHANGES (above: A2AV_ERR_UNSUPPORTED).
 *  exchanges  HOST array of `count` entries; the pointer arrays they name are
 *             read during the call only.
 *
 * The grid is divided among the exchanges in proportion to their bytes
 * (each gets at least one CTA).  Engine: vector when the handle's path is
 * A2AV_PATH_VECTOR or any buffer of the call is outside device memory; bulk
 * when every row and buffer of every exchange is 16-byte aligned (path AUTO
 * or BULK); staged otherwise.  Memory rules as for
 * a2av_run, across all the exchanges: no output may overlap any input,
 * split matrix or other output of the call.  Validity is checked per
 * exchange: one with invalid splits writes nothing of its own (no output
 * byte, no out_splits_offsets entry) and records A2AV_ERR_BAD_SPLITS; the
 * others are carried out.  Host errors as for a2av_run (any entry), plus
 * A2AV_ERR_INVALID_ARG for count < 1 or exchanges == NULL.
 */
int a2av_run_multi(a2av_handle *h, int count, const a2av_exchange_t *exchanges, void *stream);

/*
 * a2av_status -- read and clear the handle's device status word: the first
 * device-detected error (A2AV_ERR_BAD_SPLITS, A2AV_ERR_TIMEOUT or
 * A2AV_ERR_BAD_INDEX) of the runs
 * since the last call, or A2AV_OK.  Enqueues a 4-byte device-to-host copy and
 * a reset on `stream` and synchronizes that stream: the only host round trip
 * of the library.  `device_status` is a host pointer.
 * Errors: A2AV_ERR_INVALID_ARG, A2AV_ERR_CUDA.
 */
int a2av_status(a2av_handle *h, void *stream, int *device_status);

/*
 * a2av_destroy -- free the handle and its status word.  Work already
 * enqueued must have finished (synchronize its stream first).  NULL is a
 * no-op returning A2AV_OK.
 */
int a2av_destroy(a2av_handle *h);

/*
 * a2av_set_path -- choose the copy engine for later runs (a2av_path_t).
 * A2AV_PATH_BULK on a run whose row_bytes or buffer addresses are not all
 * 16-byte aligned falls back to the staged engine for that run; a run with
 * any buffer outside device memory takes the vector engine (a2av_run).
 * Also forgets the handle's remembered pointer classifications.
 * Errors: A2AV_ERR_INVALID_ARG.
 */
int a2av_set_path(a2av_handle *h, int path);

/*
 * a2av_set_grid -- CTAs launched per SM for later runs (1..32; 0 restores
 * the engine's default).  Errors: A2AV_ERR_INVALID_ARG.
 */
int a2av_set_grid(a2av_handle *h, int ctas_per_sm);

/*
 * a2av_last_launch -- describe the most recent successful a2av_run of this
 * handle: the engine used (a2av_path_t, never AUTO), the grid size and the
 * threads per CTA.  Any output pointer may be NULL.
 */
int a2av_last_launch(const a2av_handle *h, int *path, int *grid, int *block);

/*
 * a2av_last_dispatch -- describe the most recent successful a2av_dispatch or
 * a2av_combine_items of this handle: the number of kernels it enqueued, the
 * number of workspace memsets before them (0 or 1) and the name of the
 * kernel that moved the rows (a static string, "" before the first call).
 * Any output pointer may be NULL.  Errors: A2AV_ERR_INVALID_ARG (h == NULL).
 */
int a2av_last_dispatch(const a2av_handle *h, int *kernels, int *memsets, const char **copy_kernel);

/* a2av_error_string -- a static English description of a status code. */
const char *a2av_error_string(int code);

/* a2av_version -- 10000*major + 100*minor + patch of this library. */
int a2av_version(void);

/* Bytes of device memory the library reserves for a2av_run_noalloc. */
#define A2AV_NOALLOC_SCRATCH_BYTES 256

/* Device workspace a2av_combine_items needs (flag and an offsets table). */
#define A2AV_COMBINE_WORKSPACE_BYTES (256 + 16 * A2AV_MAX_RANKS * A2AV_MAX_RANKS)

/*
 * a2av_combine_items -- the fused combine: the return path of a2av_dispatch
 * with every row put straight back in item order.  The pages' MoE region
 * (PR 154580) sends tokens to their experts and back; the plain reverse
 * exchange (a2av_combine) returns each rank its rows in key order, which
 * the caller would then permute by sorted_pos -- a second read and write of
 * every row that this call does not make.
 *
 * After a2av_dispatch with keys_per_peer K, S = its in_splits_dev, and
 * sorted_pos and keys as it took and returned them, peer p holds, in the
 * layout the dispatch wrote out[p], a row for each of its items (e.g. an
 * expert's output rows).  For every rank r and item i, with p = key / K:
 *   item_out[r][i] = peer[p] row (out_off[p][r] + sorted_pos[r][i] - in_off[r][p])
 * (offsets of S as in a2av_run): combine_items(dispatch(x)) puts every
 * item's source row back at its item index.
 *
 *  peer_ptrs          HOST array of W device pointers: peer p's rows in the
 *                     dispatch layout (sum_r S[r][p] rows).  Read only.
 *  in_splits_dev      DEVICE int64 [W][W]: S as a2av_dispatch wrote it.
 *  key_ptrs, sorted_pos_ptrs, items_per_rank: as a2av_dispatch took and
 *                     wrote them (HOST arrays of W device int32 / int64
 *                     arrays, HOST int64 counts).  Read only.
 *  item_out_ptrs      HOST array of W device pointers: rank r's items_per_rank[r]
 *                     rows, written in item order.
 *  workspace          DEVICE scratch, 256-byte aligned, at least
 *                     A2AV_COMBINE_WORKSPACE_BYTES, not shared with a call in flight.
 *
 * Launches (a2av_last_dispatch reports which): at most 4096 items over all
 * ranks -- ONE kernel, no workspace memset (every block checks the split
 * matrix and every key and position, then copies its share); otherwise a
 * 256-byte workspace memset, then (A2AV_DISPATCH_ORDER at a2av_create
 * above 0) for rows shorter than 64 bytes ONE cooperative kernel that
 * checks every item, passes a grid barrier and copies, and for 16-byte
 * aligned device rows of 64 bytes to 2 KiB the cp.async.bulk gather,
 * launched cooperatively, which checks every item itself before a grid
 * barrier and stores no row before every block has arrived there; else a
 * check kernel (the split matrix, each key, each position
 * within its destination's group) and then the dispatch's copy kernel with
 * the rows moving the other way.  The grid barriers are bounded (about a
 * second, then A2AV_ERR_TIMEOUT).  Device errors A2AV_ERR_BAD_SPLITS (as
 * a2av_run; NULL buffers with rows) and A2AV_ERR_BAD_INDEX (a key outside
 * [0, W * K) or a position outside [in_off[r][p], in_off[r][p] + S[r][p]))
 * write nothing.  Host errors as a2av_dispatch (A2AV_ERR_INVALID_ARG also
 * for a small or misaligned workspace).
 */
int a2av_combine_items(a2av_handle *h, int keys_per_peer, const void *const *peer_ptrs,
                       const int64_t *in_splits_dev, const int32_t *const *key_ptrs,
                       const int64_t *const *sorted_pos_ptrs, const int64_t *items_per_rank,
                       void *const *item_out_ptrs, int64_t row_bytes, void *workspace,
                       int64_t workspace_bytes, void *stream);

/*
 * a2av_run_noalloc -- the same exchange as a2av_run, for callers that cannot
 * allocate device memory.  (The pages have no counterpart; this is an
 * interface addition of this library.)
 *
 * Who needs it: a2av_create calls cudaMalloc for the handle's status word.
 * Some callers may not do that: engines that plan every byte of device memory
 * up front and forbid allocation once they run, hosts that own the only
 * allocator and hand plug-ins nothing but buffers, and code on a latency path
 * where cudaMalloc's implicit device synchronisation is not acceptable.  This
 * entry point takes no handle and allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.  The caller still passes every
 * input and output.
 *
 * Scratch: the status word lives in a fixed A2AV_NOALLOC_SCRATCH_BYTES-byte
 * array inside the library's own device code.  Every GPU that loads the
 * library holds that array until the process exits.  Each call clears the
 * status word on `stream` before its kernel runs.  All calls in the process
 * share the one array: calls whose work overlaps on the GPU (different
 * streams, or different host threads) race on it, so their statuses are not
 * reliable; serialise such calls.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and configures the kernels, with that device
 * current.  Make that first call before any stream capture begins.  The
 * set-up is kept for the life of the process: a cudaDeviceReset (or any
 * other teardown of the device's primary context) invalidates it, so do not
 * call this entry point on a device after resetting it.
 *
 * Arguments: world_size, in_capacity_rows and out_capacity_rows as in
 * a2av_create; in_ptrs .. stream as in a2av_run (the copy engine is chosen as
 * A2AV_PATH_AUTO does).  device_status: NULL makes the call asynchronous like
 * a2av_run, with no status reported; a host int* makes the call wait for the
 * exchange (it synchronises `stream`) and store the device-detected status
 * there (A2AV_OK, A2AV_ERR_BAD_SPLITS or A2AV_ERR_TIMEOUT).
 *
 * Limit: the scratch does not grow with the exchange, so the only size the
 * call can exceed is the rank count.  world_size > A2AV_MAX_RANKS returns
 * A2AV_ERR_UNSUPPORTED; a device ordinal of 64 or more also returns
 * A2AV_ERR_UNSUPPORTED.  Other host errors are those of a2av_run.
 */
int a2av_run_noalloc(int world_size, int64_t in_capacity_rows, int64_t out_capacity_rows,
                     const void *const *in_ptrs, const int64_t *in_splits_dev,
                     void *const *out_ptrs, int64_t *out_splits_offsets_dev, int64_t row_bytes,
                     void *stream, int *device_status);

#ifdef __cplusplus
}
#endif

#endif /* A2AV_H_ */
