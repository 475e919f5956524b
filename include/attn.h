/*
 * attn.h -- C ABI of the tiled attention forward library (libattn.so).
 *
 * The library computes exact softmax attention
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 *
 * tile by tile with the online-softmax running statistics: the row max m,
 * the exp-sum l relative to m, the value accumulator u weighted the same
 * way, and the rescale factor r = exp(m_old - m_new) applied to l and u
 * whenever m grows (page S23-J17, clxhxhhr.top/posts/5544, §3.1 "在线
 * Softmax 只需三个量"; the same recurrence in normalised form is the
 * online-softmax pseudocode of the ans20xx.com day14 page).  The L x L score
 * and probability matrices never reach global memory: only O and the per-row
 * log-sum-exp leave the kernel (S23-J17 §3 accounts the 1 GiB of S/P traffic
 * this avoids at L = 8192, d = 128).
 *
 * Problem statement (lei6393.com flash-attention training-integration page):
 *   - multi-head and grouped-query attention (§2.3: query head h reads KV
 *     head h / (Hq / Hkv), i.e. consecutive groups of Hq/Hkv query heads
 *     share one KV head);
 *   - causal or not (§2.2); causal keeps key j for query i iff
 *     j <= i + (Lk - Lq), the diagonal included;
 *   - padded batches given as packed variable-length sequences (§2.5: the
 *     key_padding_mask keeps a prefix of each row, which the MHA module
 *     unpads into a packed batch described by cumulative lengths);
 *   - softmax_scale defaults to 1/sqrt(head_dim) (§8.5); here it is always
 *     passed explicitly.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller; the library neither frees nor retains them past
 *     the call's completion on `stream`.
 *   - Work is enqueued on `stream`; no entry point except attn_get_error()
 *     synchronises.  Arguments are validated on the host before anything is
 *     enqueued; a non-zero return means nothing was launched.
 *   - The library allocates, per device and lazily, its own buffers: cached
 *     TMA descriptors (host memory), a device copy of the tile schedule of
 *     each dense problem shape whose schedule is too large to travel in the
 *     kernel parameters, a split-KV workspace for the forward and a D / lse
 *     workspace for the backward.  For attn_fwd: schedules are cached per
 *     shape, at most 256 per kernel; the least recently used one is evicted
 *     and its device copy released with cudaFreeAsync on the calling stream,
 *     ordered after every launch that read it.  A schedule is written to the
 *     device by a kernel on the calling stream (its values in the launch
 *     parameters), so the first call of a shape neither synchronises nor
 *     copies from pageable memory, and it may be made inside a stream
 *     capture.  The forward's workspaces grow with cudaMallocAsync; the
 *     buffer they replace is released with cudaFreeAsync on the calling
 *     stream.  Schedules and workspaces that a captured graph uses are kept
 *     until the process exits (a replay reads them).
 *   - Calls that share a device may run concurrently on different streams,
 *     except that each workspace is one buffer per device: at most one
 *     forward whose schedule splits the keys (attn_plan reports partials > 0;
 *     varlen calls never split) and at most one backward may be in flight on
 *     a device at a time.  Order such calls (one stream, or events).
 */
#ifndef ATTN_H
#define ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *cudaStream_t;

/* ---- return codes ------------------------------------------------------ */
#define ATTN_OK 0
#define ATTN_EINVAL (-1)       /* bad argument: null pointer, non-positive size, Hq % Hkv != 0,
                                  pointer not 16-byte aligned, size out of range */
#define ATTN_EUNSUPPORTED (-2) /* valid but not built: head_dim other than 64 or 128, or a
                                  device that is not sm_103 */
#define ATTN_ELAUNCH (-3)      /* a CUDA runtime or driver call failed */
#define ATTN_ENOMEM (-4)       /* the library could not allocate its workspace */
#define ATTN_EDEVICE (-5)      /* returned by attn_get_error(): a kernel reported an error */
#define ATTN_ETOOLARGE (-6)    /* attn_fwd_noalloc only: the problem's schedule or split-KV
                                  partials exceed its static scratch buffer */

/* Device-side error codes, reported through attn_get_error() (as
 * ATTN_EDEVICE) and readable with attn_last_device_error(). */
#define ATTN_DEVERR_WAIT_TIMEOUT 0x100  /* a pipeline barrier wait ran past its time limit;
                                           low byte names the wait site */
#define ATTN_DEVERR_BAD_SEQLENS 0x200   /* cu_seqlens not non-decreasing from 0, or its last
                                           entry exceeds the packed length */

/*
 * attn_fwd -- attention forward, bf16 inputs and outputs, fp32 accumulation.
 *
 *   q    (B, Lq, Hq, d) bf16, contiguous            [dense]
 *        (Lq, Hq, d) packed rows                    [varlen, cu_seqlens != NULL]
 *   k, v (B, Lk, Hkv, d) bf16, contiguous           [dense]
 *        (Lk, Hkv, d) packed rows                   [varlen]
 *   o    same shape and dtype as q; written
 *   lse  float32 log-sum-exp of the scaled scores (natural log), written:
 *        (B, Hq, Lq) [dense] or (Hq, Lq) indexed by packed row [varlen].
 *        A row that sees no key gets O = 0 and lse = -inf.
 *   B, Hq, Hkv   batch (number of sequences for varlen), query heads and KV
 *                heads; Hq must be a multiple of Hkv.
 *   Lq, Lk       dense: query and key length of every sequence.
 *                varlen: number of packed rows in q/o and in k/v (the
 *                buffers' extents); self-attention only, so Lq == Lk.
 *   d            head_dim, 64 or 128.
 *   causal       0 or 1 (mask described above; for varlen it applies within
 *                each sequence).
 *   scale        softmax scale applied to Q K^T (usually 1/sqrt(d)); finite.
 *   cu_seqlens_or_null
 *                NULL for dense inputs; else a DEVICE int32 array of B+1
 *                cumulative sequence lengths, cu[0] = 0, non-decreasing,
 *                cu[B] <= Lq, shared by queries and keys.  The host never
 *                reads it; a malformed array is reported through
 *                attn_get_error() and its rows are left unwritten.
 *   stream       CUDA stream to enqueue on (NULL = legacy default stream).
 *
 * All of q, k, v, o must be 16-byte aligned and lse 4-byte aligned.
 * Returns ATTN_OK or a negative code; see attn_strerror().
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
             float scale, const int *cu_seqlens_or_null, cudaStream_t stream);

/* attn_fwd_fp16 -- the same operation and argument rules with fp16 q, k, v
 * and o (the SDPA experiment of the ans20xx.com day14 page, 实验 2, runs in
 * float16). */
int attn_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                  float scale, const int *cu_seqlens_or_null, cudaStream_t stream);

/*
 * attn_fwd_noalloc -- attn_fwd (bf16) for callers that cannot allocate
 * device memory.  The paper has no counterpart: this is a deployment
 * variant of the same operation, not part of the method.
 *
 * attn_fwd allocates on first use of a problem shape (its schedule) and
 * grows a split-KV workspace with cudaMalloc/cudaFree.  Some callers cannot
 * allow that: a process whose device memory is owned by a pool or caching
 * allocator that has already reserved it (a surprise cudaMalloc may fail),
 * or a latency-critical loop where cudaFree's implicit device-wide
 * synchronisation would stall every other stream.  This entry point takes
 * the same arguments and performs the same computation with the same
 * kernels, but its scratch (the schedule and the split-KV partials) lives in
 * one file-scope device array of ATTN_NOALLOC_SCRATCH_BYTES (24 MiB: 4 MiB
 * for the schedule, 20 MiB for partials) that every GPU loading the library
 * holds until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero (every partial is written
 *     before it is read).  A schedule too large for the launch parameters
 *     is written into the array on every call, by a small kernel on
 *     `stream` ahead of the attention kernels.  Calls whose work overlaps on the GPU (for example
 *     on two streams without an ordering between them) race on the array and
 *     give wrong results: order them.
 *   - A dense problem whose schedule exceeds 4 MiB or whose partials exceed
 *     20 MiB returns ATTN_ETOOLARGE without launching anything; use attn_fwd.
 *     Varlen calls use no scratch.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (24u << 20)
int attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                     float scale, const int *cu_seqlens_or_null, cudaStream_t stream);

/*
 * attn_fwd_varlen -- the packed (varlen) forward with separate query and key
 * offsets: cross-attention between packed batches, and queries that extend a
 * key/value cache (training page §2.4 cross-attention; §4, rotary offsets
 * from the cache length during generation).  q, o are (total_q, Hq, d), k, v
 * are (total_k, Hkv, d); sequence b has queries cu_seqlens_q[b] ..
 * cu_seqlens_q[b+1] - 1 and keys cu_seqlens_k[b] .. cu_seqlens_k[b+1] - 1 (both
 * device int32 arrays of B+1 entries, 0 first, non-decreasing, last entry
 * at most the total; checked by the kernel as for attn_fwd; rows past the
 * last sequence, up to the next 128-row boundary, are loaded with whole tiles
 * and weighted by zero, so they must hold finite values).  Causal aligns
 * bottom-right per sequence: query i of a sequence with Lq_b queries and Lk_b
 * keys sees key j iff j <= i + Lk_b - Lq_b (the queries are the last Lq_b
 * positions, as when a cache of Lk_b - Lq_b tokens precedes them); a query
 * that sees no key gives O = 0, lse = -inf.  lse is (Hq, total_q).  fp16 = 0
 * selects bf16 tensors, 1 fp16.  B <= 4096.  Return codes as attn_fwd.
 *
 * Grouped heads: when Hq / Hkv is a power of two from 2 to 32, every packed
 * forward (this entry point and attn_fwd with cu_seqlens) lets the query
 * heads of one key/value head share a tile: 128 / group positions x group
 * heads instead of 128 positions of one head.  Each key/value tile is then
 * read once per group, and a sequence with one new token (decoding) fills
 * group rows of a tile instead of one.  Every output row is the same
 * function of its inputs either way.
 *
 * Scheduling: the kernel builds its work list from the offsets on the
 * device.  With separate key offsets, up to 32 sequences whose key counts
 * differ by more than 4x are numbered by key count (most first) and the work
 * units placed on the CTAs in snake order, so long and short units share
 * CTAs; otherwise the units go round-robin in sequence order.  The results do
 * not depend on the placement.
 */
int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                    int total_q, int total_k, int d, int causal, float scale, const int *cu_seqlens_q,
                    const int *cu_seqlens_k, int fp16, cudaStream_t stream);

/*
 * attn_decode -- one decoding step: a single new query per sequence against
 * the sequence's key/value cache (training page §4, generation with a cache
 * whose length sets the rotary offset; the same exact softmax of page
 * S23-J17, clxhxhhr.top/posts/5544, §3.1, reached by splitting the keys into
 * chunks and merging the chunks with the running-max rescaling).  The result
 * is that of attn_fwd_varlen with cu_seqlens_q = {0, 1, ..., B}: the query is
 * the last position of its sequence, so causal and non-causal coincide and it
 * sees all of the sequence's keys.
 *
 *   q, o  (B, Hq, d) contiguous, one row per sequence;
 *   k, v  (total_k, Hkv, d) contiguous, sequence b holding rows
 *         cu_seqlens_k[b] .. cu_seqlens_k[b+1] - 1 (a device int32 array of
 *         B+1 entries, 0 first, non-decreasing, last entry at most total_k;
 *         checked on the device: a malformed array records
 *         ATTN_DEVERR_BAD_SEQLENS and every row gets O = 0, lse = -inf);
 *   lse   (Hq, B) float32, natural log; a sequence with no key gives O = 0
 *         and lse = -inf.
 *
 * fp16 = 0 selects bf16 tensors, 1 fp16.  d is 64 or 128 and Hq / Hkv is 1,
 * 2, 4 or 8 (else ATTN_EUNSUPPORTED; attn_fwd_varlen takes the others).
 * Pointers 16-byte aligned (lse 4); k and v may be null when total_k is 0.
 *
 * Two routes compute it (attn_set_decode_path).  The default runs on TMA
 * tiles and tcgen05 MMAs, reading the cache once per key/value head: a
 * decode kernel with the products transposed (S^T = K Q^T, u^T += V^T P^T:
 * the tile's 128 keys on the TMEM lanes, the group's query heads on the
 * columns, so each softmax thread owns one key); at head_dim 64 each softmax
 * step takes two key tiles.  With head_dim 64 and more than 3143 sequences
 * the packed forward kernel in decode mode (the group's query heads in one
 * tile) runs instead.  Units are (sequence, key/value head, piece of the cache): the
 * caches are cut into pieces of key tiles when that shortens the step (a
 * cost model over rounds of one unit per SM, with the mean cache length),
 * and a second launch merges the pieces' fp32 partials with the running-max
 * rescaling; partials live in the library's stream-ordered split workspace.  The
 * other route runs on the CUDA cores: a one-warp pass over cu_seqlens_k, one
 * block per chunk of 128 keys and key/value head, and a merge per (sequence,
 * query head), with the chunk results in a workspace grown with cudaMalloc
 * (calls that overlap on the GPU must not share a device); calls with
 * total_k = 0 or B > 4096 always take it.  Returns ATTN_OK, ATTN_EINVAL,
 * ATTN_EUNSUPPORTED, ATTN_ENOMEM or ATTN_ELAUNCH.
 */
int attn_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
                int total_k, int d, float scale, const int *cu_seqlens_k, int fp16, cudaStream_t stream);

/*
 * attn_bwd -- the backward of the dense forward: the gradients of
 * sum(dout * O) with respect to q, k and v (training page §5.3: the backward
 * recomputes the attention weights from what the forward kept, and nothing
 * of size L x L is stored).  With P_ij = exp(scale q_i.k_j - lse_i) (the
 * forward's weights, recomputed from its lse), dP_ij = dout_i . v_j and
 * D_i = dout_i . O_i:
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dout_i
 * with the sums over the keys j that query i sees (the forward's causal
 * rule) and, for dk and dv, over the query heads that share the KV head.
 *
 * q, o, dout, dq: (B, Lq, Hq, d); k, v, dk, dv: (B, Lk, Hkv, d); all
 * contiguous 16-bit (fp16 = 0: bf16, 1: fp16), 16-byte aligned device
 * pointers.  lse: (B, Hq, Lq) fp32 as attn_fwd returns it (a row with
 * lse = -inf gets no gradient).  o and lse must be the forward's outputs for
 * the same q, k, v, causal and scale.  dq, dk, dv are overwritten (not
 * accumulated) and must not overlap the inputs.  d in {64, 128}.  With
 * Lq = 0 the query-side pointers (q, o, lse, dout, dq) may be null and dk,
 * dv are zeroed; with Lk = 0 the key-side ones (k, v, dk, dv) may be null
 * and dq is zeroed.
 *
 * The library keeps one device workspace per device (8 * B * Hq * Lq bytes,
 * rounded up), grown with cudaMalloc when a larger problem arrives.  Three
 * kernels run on `stream` (D_i, then dk and dv, then dq); the call returns
 * without waiting.  Returns ATTN_EINVAL for null or misaligned pointers and
 * bad sizes, ATTN_EUNSUPPORTED for another d or device, ATTN_ENOMEM when the
 * workspace cannot grow, ATTN_ELAUNCH on a launch failure; device-side wait
 * timeouts are reported by attn_get_error as for attn_fwd.  Varlen batches
 * are not accepted here.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
             void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
             float scale, int fp16, cudaStream_t stream);

/*
 * attn_bwd_varlen -- attn_bwd for packed batches, the backward of
 * attn_fwd_varlen (and of attn_fwd with cu_seqlens, passing the same array
 * twice).  q, o, dout, dq are (total_q, Hq, d); k, v, dk, dv (total_k, Hkv, d);
 * lse (Hq, total_q) as the varlen forward returns it; sequence b has queries
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1] - 1 and keys cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1] - 1 (device int32 arrays of B+1 entries, 0 first,
 * non-decreasing, last entry at most the total; checked on the device, a
 * malformed array is ATTN_DEVERR_BAD_SEQLENS and nothing is computed).
 * Causal aligns bottom-right per sequence as in attn_fwd_varlen.  Rows of dq,
 * dk, dv outside every sequence are left unwritten.  The workspace is
 * 8 * Hq * 128 * (B + total_q / 128 + 1) bytes plus 8 * (B + 1).  Other
 * arguments and return codes as attn_bwd.
 */
int attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                    const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int total_q,
                    int total_k, int d, int causal, float scale, const int *cu_seqlens_q,
                    const int *cu_seqlens_k, int fp16, cudaStream_t stream);

/*
 * attn_rotary -- rotary position embedding of a Q or K tensor (training
 * page §4: rotary dimension, base frequency, GPT-NeoX or GPT-J pairing, and a
 * position offset that starts new tokens at the cache length).  x and y are
 * (B, L, H, d) (dense) or packed (total, H, d) with cu_seqlens (device, B+1);
 * y may be x (in place) or a disjoint buffer (a partial overlap is
 * ATTN_EINVAL).  Token i of sequence b sits at position i + offsets[b]
 * (offsets: device int32 array of B, or null for 0).  For pair p <
 * rot_dim/2 (the features (p, p + rot_dim/2), or (2p, 2p+1) when
 * interleaved), with a = position * base^(-2p / rot_dim), (x1, x2) becomes
 * (x1 cos a - x2 sin a, x1 sin a + x2 cos a); features from rot_dim on are
 * copied.  rot_dim even, 0 < rot_dim <= d; base > 1; fp16 = 0 bf16, 1 fp16.
 * fp32 arithmetic, result rounded to the tensor's type.  Returns ATTN_OK,
 * ATTN_EINVAL or ATTN_ELAUNCH.
 */
int attn_rotary(const void *x, void *y, int B, int L, int H, int d, int rot_dim, float base, int interleaved,
                const int *cu_seqlens_or_null, int total, const int *offsets_or_null, int fp16,
                cudaStream_t stream);

/*
 * attn_rotary_packed -- the same rotation on the packed layouts the training
 * page's rotary module takes (§4.2: a packed qkv tensor (B, L, 3, H, d), whose
 * Q and K parts it rotates in place, and Q beside a packed kv tensor
 * (B, L, 2, H, d), whose K part it rotates).  Every token row holds h_total
 * heads of d features (3H for qkv, 2H for kv); the first h_rot of them are
 * rotated (2H for qkv, H for kv).  In place (y == x) the other heads are left
 * alone; out of place they are copied to y.  Other arguments, layouts and
 * return codes as attn_rotary; 0 < h_rot <= h_total.
 */
int attn_rotary_packed(const void *x, void *y, int B, int L, int h_total, int h_rot, int d, int rot_dim,
                       float base, int interleaved, const int *cu_seqlens_or_null, int total,
                       const int *offsets_or_null, int fp16, cudaStream_t stream);

/*
 * Padded batches around the varlen forward (the flash-attention
 * training-integration page, §2.5: drop the padded positions, run the
 * variable-length call, put the outputs back).  Each call enqueues device
 * kernels on `stream` and returns without synchronising; device pointers
 * throughout, owned by the caller.
 *
 * attn_unpad_index -- from a key-padding mask (B, L) of bytes, nonzero =
 *   keep, writes cu_seqlens (B+1 int32: cu[0] = 0, cu[b+1] = cu[b] + kept
 *   tokens of row b) and indices (B*L int32 slots: indices[cu[b] + k] =
 *   b*L + i for the k-th kept position i of row b, in order; slots from
 *   cu[B] on are left untouched).  Kept tokens need not form a prefix.
 *   Returns ATTN_EINVAL (null pointer, B or L <= 0, B*L >= 2^31) or
 *   ATTN_ELAUNCH.
 *
 * attn_gather_rows -- dst row r = src row indices[r] for r < n = min(n_max,
 *   *n_dev) (n_dev is a DEVICE int, e.g. cu_seqlens + B, so no host sync
 *   is needed; dst must hold n_max rows).  Rows n .. n+127 of dst (those
 *   below n_max) are set to zero: the attention kernels load whole 128-row
 *   tiles, so the rows just past the last sequence are read (and weighted by
 *   zero, which needs them finite).  Rows are row_bytes long (a multiple of
 *   16); src has src_rows rows and an index outside [0, src_rows) moves
 *   nothing.  src and dst 16-byte aligned.
 *
 * attn_scatter_rows -- dst row indices[r] = src row r for r < min(n_max,
 *   *n_dev); dst has dst_rows rows (indices outside are skipped) and its
 *   other rows are left as they are (fill them first, e.g. with zeros).
 *
 * attn_scatter_lse -- lse of a varlen call, (Hq, n_max) fp32 (n_max = the
 *   packed row count passed to attn_fwd), to the padded (B, Hq, L):
 *   dst[b, h, i] = src[h, r] where indices[r] = b*L + i, r < min(n_max,
 *   *n_dev); other entries left as they are (fill with -inf first).
 *
 * The three return ATTN_OK, ATTN_EINVAL (null pointer, negative count,
 * row_bytes not a positive multiple of 16, misaligned row pointer, or a
 * padded extent of 2^31 rows or more) or ATTN_ELAUNCH.
 */
int attn_unpad_index(const unsigned char *mask, int B, int L, int *cu_seqlens, int *indices, cudaStream_t stream);
int attn_gather_rows(const void *src, int src_rows, const int *indices, int n_max, const int *n_dev, int row_bytes,
                     void *dst, cudaStream_t stream);
int attn_scatter_rows(const void *src, const int *indices, int n_max, const int *n_dev, int row_bytes, void *dst,
                      int dst_rows, cudaStream_t stream);
int attn_scatter_lse(const float *src, const int *indices, int n_max, const int *n_dev, int Hq, int B, int L,
                     float *dst, cudaStream_t stream);

/*
 * attn_set_pair_forward -- selects the kernel of dense head_dim-128 forwards
 * (attn_fwd, attn_fwd_fp16): 1 runs them on CTA pairs, where one tcgen05
 * .cta_group::2 MMA spans two SMs (256 query rows against 256 keys) and split
 * key ranges are merged inside the kernel; 0 (the default) runs them on the
 * single-CTA kernel with a separate merge pass.  Both compute the same
 * function.  attn_pair_forward_used(d, varlen) tells which one attn_fwd takes
 * (1: the pair kernel).  Process-wide; not synchronised with calls in flight.
 */
void attn_set_pair_forward(int enable);
int attn_pair_forward_used(int d, int varlen);

/*
 * attn_set_cluster_merge -- how dense forwards on the single-CTA kernel merge
 * split key ranges (the r = exp(m_s - M) rescaling of page S23-J17 §3.1,
 * applied across pieces).  0 (the default): the host plans
 * pieces of any length where they balance the load, the pieces write fp32
 * partials to a workspace and a separate combine pass merges them.  2, 4 or
 * 8: every 256-row query block is split into that many pieces of equal key
 * ranges, the pieces of a block run as one thread-block cluster, keep their
 * partials in shared memory and merge them over distributed shared memory
 * inside the kernel (no workspace, no combine pass).  Both compute the same
 * function; the second suits shapes whose blocks all have the same key range
 * (non-causal).  Other values are ignored.  attn_cluster_merge() returns the
 * setting.  Process-wide; not synchronised with calls in flight.
 */
void attn_set_cluster_merge(int cluster_size);
int attn_cluster_merge(void);

/*
 * attn_fwd_rope -- attn_fwd of rotary-embedded queries and keys (training
 * page §4: the rotary module, rotary dimension, base frequency, GPT-NeoX or
 * GPT-J pairing, a position offset for queries that extend a cache):
 *     O = attention(rope(q, positions q_offset + i), rope(k, positions j), v)
 * with rope as attn_rotary applies it (pair i of the first rot_dim features
 * rotated by position * base^(-2 i / rot_dim); interleaved = 1 pairs (2i,
 * 2i+1), 0 pairs (i, i + rot_dim/2); the rotated values rounded to the
 * tensors' 16-bit type).  q and k are read, not modified.  Dense layouts as
 * attn_fwd (no cu_seqlens); d 64 or 128; rot_dim a multiple of 16, at most d;
 * base > 1; q_offset >= 0 (Lk - Lq places the queries after a cache).
 *
 * The rotation of Q is fused into the forward kernel: each softmax thread
 * rotates its own query row in shared memory after the unit's Q block lands
 * and before its first S = Q K^T, from a (cos, sin) table the library keeps
 * (computed once per rotary dimension, base and position count, with the
 * rotary pass's arithmetic).  K is rotated by the rotary pass into a library
 * workspace first: a key tile is loaded once per query block, so rotating it
 * in the tile load would repeat the rotation L / 256 times per key.  Two or
 * three launches on `stream` (table when new, rotary of K, forward (+ merge));
 * workspaces are stream-ordered like attn_fwd's.  Return codes as attn_fwd.
 * Measured on the GB300: the rotation at every unit start delays the unit's
 * first MMA, so attn_rotary on q and k followed by attn_fwd is faster (e.g.
 * 44.7 against 48.8 us for one head of 8192 causal tokens at d 128).
 */
int attn_fwd_rope(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Lq,
                  int Lk, int d, int causal, float scale, int rot_dim, float base, int interleaved, int q_offset,
                  int fp16, cudaStream_t stream);

/*
 * attn_set_decode_path -- selects how attn_decode runs: 1 (the default) on
 * tensor cores, the transposed decode kernel (the query heads of a
 * key/value head are the MMA's columns, and each cache is cut into pieces of
 * key tiles, merged by a second pass, when the (sequence, head group) units
 * alone would leave SMs idle); 0 on the CUDA-core chunk kernels.  Both
 * compute the same function.  Calls with total_k = 0 or B > 4096 take the
 * CUDA-core path either way.  attn_decode_path() returns the setting.
 * Process-wide; not synchronised with calls in flight.
 */
void attn_set_decode_path(int tensor_cores);
int attn_decode_path(void);

/*
 * attn_plan_pair -- the CTA-pair kernel's schedule for a dense problem, for
 * inspection and tests (no GPU needed).  Units as attn_plan's, with m_block a
 * 256-row query block (128 rows in each CTA of the pair), [kv_begin, kv_end)
 * counted in 256-key tiles and `cta` the pair that runs the unit;
 * *n_pairs receives the number of pairs (the grid is twice that).
 */
int attn_plan_pair(int B, int Hq, int Hkv, int Lq, int Lk, int causal, int num_pairs, int *units, int max_units,
                   int *n_units, int *n_pairs, int *n_partials);

/* attn_cache_stats -- the number of schedules cached on the current device
 * (both kernels) and how many of them a stream capture pinned. */
int attn_cache_stats(int *plans, int *pinned);

/* attn_selftest_plan_cache -- runs the schedule cache's eviction policy on
 * host-side entries only (no device memory): n_keys lookups cycling over
 * 2 * capacity + 7 keys, every pin_every-th new entry pinned (0: none).
 * Reports the largest number of live entries and how many were released. */
int attn_selftest_plan_cache(int n_keys, int capacity, int pin_every, int *max_live, int *released);

/* attn_get_error -- synchronises `stream`, then returns ATTN_EDEVICE if any
 * kernel of this library on the current device has reported an error since
 * the last call (and clears it), ATTN_ELAUNCH if the stream itself failed,
 * else ATTN_OK. */
int attn_get_error(cudaStream_t stream);

/* attn_last_device_error -- the device error code (ATTN_DEVERR_*) that the
 * last attn_get_error() call cleared, or 0. Host-only, no synchronisation. */
int attn_last_device_error(void);

/* attn_strerror -- static text for a return code. */
const char *attn_strerror(int code);

/* attn_set_wait_timeout_ns -- time limit of every pipeline barrier wait in
 * the kernels launched afterwards by this process (default 2e9 ns).  A wait
 * that runs out records ATTN_DEVERR_WAIT_TIMEOUT and the kernel returns
 * early with its outputs incomplete.  Values below 1000 are raised to 1000. */
void attn_set_wait_timeout_ns(unsigned long long ns);

/* attn_selftest_wait_timeout -- launches one CTA that waits on a barrier no
 * thread ever arrives on, under the current time limit, so that the
 * failure path (error word, early exit) can be checked on a GPU without a
 * fault or a hang.  Returns ATTN_OK if the launch was enqueued; the caller
 * then expects attn_get_error() to return ATTN_EDEVICE. */
int attn_selftest_wait_timeout(cudaStream_t stream);

/*
 * attn_plan -- the host-side persistent-kernel schedule for a dense problem,
 * exposed for inspection and tests (no GPU needed).  Writes up to
 * `max_units` work units to `units` as 8 ints each:
 *     { b*Hq + h, m_block, kv_begin, kv_end, split, n_split, partial_slot, cta }
 * where m_block indexes 256-row query blocks, [kv_begin, kv_end) is the
 * range of 128-key tiles the unit covers, split/n_split identify a split-KV
 * piece (n_split = 1: no split), partial_slot is its workspace slot (-1 if
 * none) and cta the persistent CTA that runs it.  `*n_units` receives the
 * unit count, `*n_ctas` the grid size and `*n_partials` the number of
 * workspace slots.  Returns ATTN_OK, ATTN_EINVAL, or ATTN_ENOMEM if
 * max_units is too small (then *n_units still holds the required count).
 */
int attn_plan(int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal, int num_sms,
              int *units, int max_units, int *n_units, int *n_ctas, int *n_partials);

/* attn_launch_count -- number of kernels this library has launched in this
 * process (all devices), counted on the host at each successful launch. */
unsigned long long attn_launch_count(void);

/*
 * attn_trace_enable -- phase trace of the forward kernel, for performance
 * analysis.  Trace points are compiled only into the traced build of the
 * library (libattn_trace.so, built with ATTN_TRACE=1) so that the default
 * kernels carry none of their cost; the default build returns
 * ATTN_EUNSUPPORTED.  With a non-null DEVICE buffer, every later forward
 * launch records, per CTA, four event streams (TMA producer, MMA issuer, and
 * one thread of each softmax warpgroup) of up to `events_per_stream` events.
 * An event is two 64-bit words: a tag word (tag << 56 | sub-tile << 48 |
 * unit << 24 | key tile) and the SM clock.  CTA c, stream s starts at word
 * (c * 4 + s) * events_per_stream * 2; the buffer must hold
 * grid * 4 * events_per_stream * 16 bytes, grid being at most the SM count.
 * The caller owns the buffer and keeps it alive while traced launches run.
 * A null buffer (or events_per_stream <= 0) turns tracing off.  Returns
 * ATTN_OK, ATTN_EINVAL (buffer not 16-byte aligned) or ATTN_EUNSUPPORTED.
 */
int attn_trace_enable(void *dev_buf, int events_per_stream);

/*
 * Per-call kernel timing, for benchmarks.  attn_profile_enable(n) makes the
 * next n forward calls on any stream record CUDA events around their kernels:
 * before the main kernel, after it, and after the split-KV combine (when one
 * runs).  attn_profile_read() synchronises on the recorded events and writes,
 * for up to `max` recorded calls, the main kernel's duration and the whole
 * call's duration in milliseconds; *n receives the number of calls recorded.
 * Enabling again discards earlier records.  Returns ATTN_OK, ATTN_ENOMEM or
 * ATTN_ELAUNCH.
 */
int attn_profile_enable(int n);
int attn_profile_read(float *main_ms, float *call_ms, int max, int *n);
void attn_profile_disable(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
