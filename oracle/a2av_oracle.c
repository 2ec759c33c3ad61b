/*
 * a2av_oracle.c -- plain CPU oracle for the variable-size all-to-all with
 * device-resident splits (all_to_all_vdev).
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library's product path never
 * does, and it shares no code, header or constant with the CUDA path.
 *
 * What it computes ("[a2av] Improve tuning for 4 GPUs", pytorch PR 154580,
 * section "Problem": nvshmem_all_to_all_vdev, each rank sending a
 * variable-size chunk to every peer, split sizes resident on the device):
 *
 *   W ranks.  S[r][p] = in_splits[r*W + p] >= 0 rows go from rank r to peer p.
 *   Rank r's input holds its chunks back to back in peer order, so the chunk
 *   for p starts at row in_off[r][p] = sum_{q<p} S[r][q].
 *   Peer p's output holds the chunks it receives back to back in source-rank
 *   order, so rank r's chunk lands at row out_off[p][r] = sum_{q<r} S[q][p].
 *   out_splits_offsets[p][0][r] = S[r][p]        (the transposed splits)
 *   out_splits_offsets[p][1][r] = out_off[p][r]  (their exclusive scan, rows)
 *
 * A row is row_bytes bytes; the exchange copies bytes and never looks at
 * their values.  Rows of an input past its last chunk are never read; bytes
 * of an output past its last received row are never written.
 *
 * Split validity (the pages do not say; this is the reading both sides
 * implement): every S[r][p] >= 0; S[r][p] <= 2^62 / (W * row_bytes) so that
 * every byte offset fits in a signed 64-bit integer; sum_p S[r][p] <= the
 * input capacity and sum_r S[r][p] <= the output capacity when that capacity
 * is nonzero; a NULL buffer has capacity zero.  Invalid splits leave every
 * output and out_splits_offsets untouched.
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_INVALID_ARG (-1)
#define ORACLE_BAD_SPLITS (-4)
#define ORACLE_BAD_INDEX (-6)

/* Largest byte count the exchange accepts: 2^62. */
static const int64_t kMaxBytes = (int64_t)1 << 62;

/* Rows rank r sends in total: sum over peers of S[r][q]. */
static int64_t rows_sent(int W, const int64_t *S, int r) {
  int64_t total = 0;
  for (int q = 0; q < W; ++q) total += S[(int64_t)r * W + q];
  return total;
}

/* Rows peer p receives in total: sum over sources of S[q][p]. */
static int64_t rows_received(int W, const int64_t *S, int p) {
  int64_t total = 0;
  for (int q = 0; q < W; ++q) total += S[(int64_t)q * W + p];
  return total;
}

/* in_off[r][p]: the first row of rank r's chunk for peer p. */
static int64_t in_offset(int W, const int64_t *S, int r, int p) {
  int64_t off = 0;
  for (int q = 0; q < p; ++q) off += S[(int64_t)r * W + q];
  return off;
}

/* out_off[p][r]: the first row of peer p's output that rank r's chunk fills. */
static int64_t out_offset(int W, const int64_t *S, int p, int r) {
  int64_t off = 0;
  for (int q = 0; q < r; ++q) off += S[(int64_t)q * W + p];
  return off;
}

/* Validity of the splits, as stated in the header comment.  in/out may be
 * NULL as arrays (then no buffer is NULL). */
int a2av_oracle_check(int W, const int64_t *in_splits, int64_t row_bytes,
                      int64_t in_capacity_rows, int64_t out_capacity_rows,
                      const void *const *in, void *const *out) {
  if (W < 1 || in_splits == NULL || row_bytes < 1) return ORACLE_INVALID_ARG;
  if (in_capacity_rows < 0 || out_capacity_rows < 0) return ORACLE_INVALID_ARG;
  const int64_t limit = kMaxBytes / ((int64_t)W * row_bytes);
  for (int64_t e = 0; e < (int64_t)W * W; ++e)
    if (in_splits[e] < 0 || in_splits[e] > limit) return ORACLE_BAD_SPLITS;
  for (int r = 0; r < W; ++r) {
    int64_t rows = rows_sent(W, in_splits, r);
    if (in_capacity_rows > 0 && rows > in_capacity_rows) return ORACLE_BAD_SPLITS;
    if (in != NULL && in[r] == NULL && rows > 0) return ORACLE_BAD_SPLITS;
  }
  for (int p = 0; p < W; ++p) {
    int64_t rows = rows_received(W, in_splits, p);
    if (out_capacity_rows > 0 && rows > out_capacity_rows) return ORACLE_BAD_SPLITS;
    if (out != NULL && out[p] == NULL && rows > 0) return ORACLE_BAD_SPLITS;
  }
  return ORACLE_OK;
}

/* Peer p's side of the exchange: fills out_p (the whole received stream) and
 * out_so_p[0][r] = S[r][p], out_so_p[1][r] = out_off[p][r].  Either output
 * may be NULL to skip it.  Does not validate; a2av_oracle does. */
int a2av_oracle_dest(int W, int p, const uint8_t *const *in, const int64_t *in_splits,
                     uint8_t *out_p, int64_t *out_so_p, int64_t row_bytes) {
  if (W < 1 || p < 0 || p >= W || in_splits == NULL || row_bytes < 1) return ORACLE_INVALID_ARG;
  for (int r = 0; r < W; ++r) {
    const int64_t n = in_splits[(int64_t)r * W + p];
    const int64_t src_row = in_offset(W, in_splits, r, p);
    const int64_t dst_row = out_offset(W, in_splits, p, r);
    if (out_so_p != NULL) {
      out_so_p[r] = n;
      out_so_p[W + r] = dst_row;
    }
    if (out_p == NULL) continue;
    for (int64_t i = 0; i < n; ++i)
      memcpy(out_p + (dst_row + i) * row_bytes, in[r] + (src_row + i) * row_bytes,
             (size_t)row_bytes);
  }
  return ORACLE_OK;
}

/* The whole exchange: every peer's output and the [W][2][W] int64
 * out_splits_offsets.  Returns ORACLE_BAD_SPLITS, writing nothing, when the
 * splits are invalid. */
int a2av_oracle(int W, const uint8_t *const *in, const int64_t *in_splits,
                uint8_t *const *out, int64_t *out_splits_offsets, int64_t row_bytes,
                int64_t in_capacity_rows, int64_t out_capacity_rows) {
  int rc = a2av_oracle_check(W, in_splits, row_bytes, in_capacity_rows, out_capacity_rows,
                             (const void *const *)in, (void *const *)out);
  if (rc != ORACLE_OK) return rc;
  for (int p = 0; p < W; ++p) {
    int64_t *so = out_splits_offsets == NULL ? NULL : out_splits_offsets + (int64_t)p * 2 * W;
    rc = a2av_oracle_dest(W, p, in, in_splits, out[p], so, row_bytes);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

/* Where row k of peer p's output comes from: the source rank *r and the row
 * *i of that rank's input.  Returns ORACLE_INVALID_ARG when k is not a
 * received row. */
int a2av_oracle_row_source(int W, const int64_t *in_splits, int p, int64_t k, int *r,
                           int64_t *i) {
  if (W < 1 || p < 0 || p >= W || k < 0 || in_splits == NULL) return ORACLE_INVALID_ARG;
  for (int q = 0; q < W; ++q) {
    const int64_t start = out_offset(W, in_splits, p, q);
    const int64_t n = in_splits[(int64_t)q * W + p];
    if (k >= start && k < start + n) {
      *r = q;
      *i = in_offset(W, in_splits, q, p) + (k - start);
      return ORACLE_OK;
    }
  }
  return ORACLE_INVALID_ARG;
}

/* The reverse exchange (the return path of a dispatch): peer p sends back to
 * rank r the S[r][p] rows it received from it.  That is the exchange above
 * with the transposed split matrix, S'[p][r] = S[r][p], read from the
 * dispatch's out_splits_offsets (row 0 of peer p's [2][W] block). */
int a2av_oracle_combine(int W, const uint8_t *const *in, const int64_t *dispatch_so,
                        uint8_t *const *out, int64_t *out_splits_offsets, int64_t row_bytes,
                        int64_t in_capacity_rows, int64_t out_capacity_rows) {
  if (W < 1 || dispatch_so == NULL) return ORACLE_INVALID_ARG;
  int64_t *St = (int64_t *)malloc(sizeof(int64_t) * (size_t)W * (size_t)W);
  if (St == NULL) return ORACLE_INVALID_ARG;
  for (int p = 0; p < W; ++p)
    for (int r = 0; r < W; ++r) St[(int64_t)p * W + r] = dispatch_so[(int64_t)p * 2 * W + r];
  const int rc = a2av_oracle(W, in, St, out, out_splits_offsets, row_bytes, in_capacity_rows,
                             out_capacity_rows);
  free(St);
  return rc;
}

/* Fused dispatch preparation: rank r's m_r items, item i naming source row
 * src_row[r][i] of rows[r] and key key[r][i] in [0, W*K), destination peer
 * key / K.  Each rank's items taken in increasing key order, ties in item
 * order, form its input for the exchange above (its chunks in peer order);
 * S[r][p] is the number of its items with destination p.  Writes the
 * exchange's outputs and out_splits_offsets, sorted_pos[r][i] = item i's
 * place in that order and, when in_splits is not NULL, S.  A key or source
 * row out of range gives ORACLE_BAD_INDEX and writes nothing. */
int a2av_oracle_dispatch(int W, int K, const uint8_t *const *rows, const int64_t *n_rows,
                         const int32_t *const *src_row, const int32_t *const *key,
                         const int64_t *n_items, uint8_t *const *out, int64_t *out_splits_offsets,
                         int64_t *const *sorted_pos, int64_t *in_splits, int64_t row_bytes,
                         int64_t out_capacity_rows) {
  if (W < 1 || K < 1 || row_bytes < 1) return ORACLE_INVALID_ARG;
  const int64_t nkeys = (int64_t)W * K;
  for (int r = 0; r < W; ++r)
    for (int64_t i = 0; i < n_items[r]; ++i)
      if (key[r][i] < 0 || key[r][i] >= nkeys || src_row[r][i] < 0 || src_row[r][i] >= n_rows[r])
        return ORACLE_BAD_INDEX;
  int64_t *S = (int64_t *)calloc((size_t)W * (size_t)W, sizeof(int64_t));
  uint8_t **sorted = (uint8_t **)calloc((size_t)W, sizeof(uint8_t *));
  int64_t **place = (int64_t **)calloc((size_t)W, sizeof(int64_t *));
  int rc = (S == NULL || sorted == NULL || place == NULL) ? ORACLE_INVALID_ARG : ORACLE_OK;
  for (int r = 0; r < W && rc == ORACLE_OK; ++r)
    for (int64_t i = 0; i < n_items[r]; ++i) S[(int64_t)r * W + key[r][i] / K] += 1;
  if (rc == ORACLE_OK)
    rc = a2av_oracle_check(W, S, row_bytes, 0, out_capacity_rows, (const void *const *)rows,
                           (void *const *)out);
  /* each rank's items in key order (counting order: every key value in turn,
   * its items in item order), rows gathered into a buffer of that order */
  for (int r = 0; r < W && rc == ORACLE_OK; ++r) {
    const int64_t m = n_items[r];
    sorted[r] = (uint8_t *)malloc((size_t)(m > 0 ? m : 1) * (size_t)row_bytes);
    place[r] = (int64_t *)malloc((size_t)(m > 0 ? m : 1) * sizeof(int64_t));
    if (sorted[r] == NULL || place[r] == NULL) {
      rc = ORACLE_INVALID_ARG;
      break;
    }
    int64_t next = 0;
    for (int64_t k = 0; k < nkeys; ++k)
      for (int64_t i = 0; i < m; ++i)
        if (key[r][i] == k) {
          memcpy(sorted[r] + next * row_bytes, rows[r] + (int64_t)src_row[r][i] * row_bytes,
                 (size_t)row_bytes);
          place[r][i] = next++;
        }
  }
  if (rc == ORACLE_OK)
    rc = a2av_oracle(W, (const uint8_t *const *)sorted, S, out, out_splits_offsets, row_bytes, 0,
                     out_capacity_rows);
  if (rc == ORACLE_OK) {
    for (int r = 0; r < W; ++r)
      for (int64_t i = 0; i < n_items[r]; ++i) sorted_pos[r][i] = place[r][i];
    if (in_splits != NULL)
      for (int64_t e = 0; e < (int64_t)W * W; ++e) in_splits[e] = S[e];
  }
  for (int r = 0; sorted != NULL && r < W; ++r) free(sorted[r]);
  for (int r = 0; place != NULL && r < W; ++r) free(place[r]);
  free(sorted);
  free(place);
  free(S);
  return rc;
}

/* The fused combine, the inverse of a2av_oracle_dispatch's row movement.
 * expert[p] holds peer p's rows in the layout the dispatch wrote out[p] (the
 * rows it received, source rank by source rank, each rank's in key order);
 * S is the dispatch's split matrix; each item (r, i) has its key (peer
 * p = key / K) and its position in rank r's key order, as the dispatch
 * returned them.  The item's row sits at row out_off[p][r] + (pos -
 * in_off[r][p]) of expert[p] (its rank's chunk starts at out_off[p][r], and
 * within the chunk the items keep their key order), and is copied to row i
 * of item_out[r].  Everything is checked before anything is written:
 * invalid S (as a2av_oracle_check, expert buffers as the outputs and item
 * buffers as the inputs) -> ORACLE_BAD_SPLITS; a key out of [0, W*K) or a
 * position outside its peer's group [in_off[r][p], in_off[r][p] + S[r][p])
 * -> ORACLE_BAD_INDEX. */
int a2av_oracle_combine_items(int W, int K, const uint8_t *const *expert, const int64_t *S,
                              const int32_t *const *key, const int64_t *const *sorted_pos,
                              const int64_t *n_items, uint8_t *const *item_out,
                              int64_t row_bytes) {
  if (W < 1 || K < 1 || row_bytes < 1) return ORACLE_INVALID_ARG;
  int rc = a2av_oracle_check(W, S, row_bytes, 0, 0, (const void *const *)item_out,
                             (void *const *)expert);
  if (rc != ORACLE_OK) return rc;
  const int64_t nkeys = (int64_t)W * K;
  for (int r = 0; r < W; ++r)
    for (int64_t i = 0; i < n_items[r]; ++i) {
      if (key[r][i] < 0 || key[r][i] >= nkeys) return ORACLE_BAD_INDEX;
      const int p = key[r][i] / K;
      const int64_t lo = in_offset(W, S, r, p);
      if (sorted_pos[r][i] < lo || sorted_pos[r][i] >= lo + S[(int64_t)r * W + p])
        return ORACLE_BAD_INDEX;
    }
  for (int r = 0; r < W; ++r)
    for (int64_t i = 0; i < n_items[r]; ++i) {
      const int p = key[r][i] / K;
      const int64_t row = out_offset(W, S, p, r) + (sorted_pos[r][i] - in_offset(W, S, r, p));
      memcpy(item_out[r] + i * row_bytes, expert[p] + row * row_bytes, (size_t)row_bytes);
    }
  return ORACLE_OK;
}
