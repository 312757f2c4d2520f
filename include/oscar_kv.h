/*
 * oscar_kv.h — C ABI of a rotated 2-bit (INT2) KV cache with a BF16 sink and
 * recent window, and of the decode attention that reads it, for NVIDIA GB300
 * (sm_103a).
 *
 * What it computes (sources are the pages describing OSCAR; page title and
 * section in brackets):
 *
 *  - kv_append: for every new token and KV head, rotate the post-RoPE key and
 *    value rows by the layer's orthogonal matrices, k' = k R_K, v' = v R_V
 *    ["OSCAR-LLAMACPP-Qwen3-4B-Thinking-2507-INT2-KV" model card, note under
 *    Files: K and V are rotated orthogonally after RoPE, inside the graph;
 *    "OSCAR-RotationZoo" card, File format: one head_dim x head_dim rotation
 *    per layer], clip the row to ratio * max|x| [model card, Run:
 *    LLAMA_KV_CLIP_RATIO, a clip of each row before it is quantised; RotationZoo, How
 *    to use: K clip 0.96, V clip 0.92], quantise each group of 128 channels
 *    along head_dim to 2-bit codes with an fp16 scale and zero [RotationZoo,
 *    Available rotations: group128 along head_dim; How to use:
 *    --kv-cache-dtype int2 --kv-cache-quant-group-size 128], and keep the
 *    first `sink` and the last `recent` tokens as BF16 [model card, Run:
 *    LLAMA_KV_HP_SINK / LLAMA_KV_HP_RECENT; hysenlabs article, What OSCAR
 *    compresses: the bulk of the cache INT2, BF16 only for the first and the
 *    latest tokens].
 *
 *  - attn_decode: one decode step of attention over that mixed cache without
 *    a separate dequantise pass [hysenlabs article, How the offline rotation
 *    is fit: one fused attention kernel over the mixed cache]: the query is rotated by
 *    R_K (the same rotation as K, so q'.k' = q.k) ["OSCAR-LLAMACPP-Gemma-4-
 *    12B-it-INT2-KV" card, Folders: applied to Q/K (and V)], softmax over all
 *    cached positions, and the value rotation is undone once at the output,
 *    o = o' R_V^T, unless the caller absorbs it [RotationZoo, How to use:
 *    SGLANG_OSCAR_ABSORB_V_ROTATION].
 *
 *  - Data-free rotation (OSCAR_FLAG_HADAMARD): for a model without calibrated
 *    rotations, K and V are rotated by the in-quant Hadamard instead
 *    [model card, Run: LLAMA_KV_NO_HADAMARD skips the in-quant Hadamard of
 *    models whose rotation is in-graph, and a base model falls back to
 *    data-free INT2; RotationZoo, How to use: HADAMARD_ORDER=128]:
 *    R_K = R_V = H, block-diagonal over the D/128 channel groups, each block
 *    the Sylvester Hadamard matrix of order 128 divided by sqrt(128)
 *    (H[i][k] = (-1)^popcount(i & k) / sqrt(128)).  The query and the output
 *    use the same H.  H is applied with an in-register fast Walsh-Hadamard
 *    transform; the R_K and R_V arguments are not read and may be NULL.
 *
 * Quantiser (the pages fix group, clip and 2-bit codes; the asymmetric
 * min/max form and the exact operation order are this library's definition):
 *   a = max_j |r_j| over the float32 rotated row; t = ratio * a;
 *   x_j = min(max(r_j, -t), t);
 *   per group of 128: mn = min x, mx = max x; s = fp16((mx - mn) / 3);
 *   z = fp16(mn); code = 0 if s == 0, else
 *   clamp(rint_half_even((x - z) * fl(1/s)), 0, 3);
 *   every step is a float32 round-to-nearest operation without FMA.
 *   Dequantised value: z + s * code.
 * Lloyd-Max levels (OSCAR_FLAG_LLOYD_MAX) [hysenlabs article, Installing
 * OSCAR and running a first Qwen3-8B calibration: an SGLANG_LLOYD_MAX switch;
 * Where OSCAR loses: results quoted at LM_RATIO=1.16]: the four levels of a
 * group are unevenly spaced like the four-level Lloyd-Max quantiser of a
 * Gaussian, level(c) = (0, rho, rho + 1, 2 rho + 1)[c], with rho = 1.16
 * rounded to float32 (the outer gaps are rho times the inner one).
 * The quantiser is as above except s = fp16((mx - mn) / span) with the float32
 * span = 2 rho + 1 (exact) and, with y = (x - z) * fl(1/s),
 * code = [y > m0] + [y > m1] + [y > m2] for the float32 midpoints m0 = rho/2,
 * m1 = rho + 1/2 (both exact) and m2 = fl(span - m0) (the float32 nearest to
 * 3rho/2 + 1): the nearest level; on a midpoint, the lower one.  Dequantised value:
 * z + s * level(code).  The bytes' layout does not change.
 *
 * Cache layout (bytes; every region starts on a 256-byte boundary; the cache
 * base pointer must be 256-byte aligned).  For layer l and role r (0 = K,
 * 1 = V) the role block starts at l * layer_bytes + r * role_bytes and holds,
 * in order:
 *   sink  [B][Hkv][S][D]    bf16   position p < S
 *   ring  [B][Hkv][W][D]    bf16   slot p mod W for the last W positions
 *   codes [B][Hkv][Ncap][D/4] u8   row p - S for every position p >= S
 *   sz    [B][Hkv][Ncap][D/128] x {fp16 scale, fp16 zero}, row p - S
 *   with Ncap = round_up(max(capacity - S, 0), 64).
 *   BF16 rows hold the round-to-nearest-even bf16 of the float32 rotated row.
 *   A code row is D/16 little-endian 32-bit words; with j the 128-channel
 *   group, word w bit b holds one channel's code:
 *     K: word 8j + 2c + i (c = 0..3, i = 0..1); for p = 0..7, kk = 4i + p/2,
 *        h = p % 2: bit 2p = channel 128j + 16kk + 2c + 8h, bit 16 + 2p =
 *        that channel + 1.
 *     V: word 8j + g (g = 0..7); bit 2n (n = 0..15) = channel 128j + 8n + g.
 *   These orders let the decode kernel feed codes straight into tensor-core
 *   fragments.
 *   K-only INT2 (OSCAR_FLAG_V_BF16) [model card, Run: a high-precision V cache
 *   type keeps V high precision, at more memory]: the K role is as above; the
 *   V role is instead
 *   full  [B][Hkv][capacity][D] bf16  row p = position p, for every position,
 *   and v_role_bytes = align256(B * Hkv * capacity * D * 2).
 *
 * Windows at decode time for a sequence of length T: sink = [0, min(S, T)),
 * ring = [max(S, T - W), T), INT2 = [S, max(S, T - W)).
 *
 * Ownership: the caller owns every buffer (cache, inputs, rotations, outputs,
 * workspace, status word); the library allocates nothing, keeps no state
 * between calls beyond per-device launch settings (and the optional per-thread
 * profiling events below), and only enqueues work on
 * the given stream (a cudaStream_t passed as void*; NULL = legacy default).
 * Calls may be captured in CUDA graphs.
 *
 * Errors: every entry point returns an oscar_status.  Argument checks happen
 * on the host before anything is launched.  Conditions only the device can see
 * are OR-ed into *dev_status (an int32 in device memory, may be NULL); kernels
 * never trap.
 */
#ifndef OSCAR_KV_H
#define OSCAR_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSCAR_KV_GROUP 128       /* quant group along head_dim */
#define OSCAR_KV_MAX_SPLITS 64   /* upper bound on decode partial slots per query head */
#define OSCAR_KV_CALIB_MAX_ROWS 268431360LL /* calibration rows per call: 65535 chunks of 4096 */

/* config flags */
enum {
  OSCAR_FLAG_ABSORB_V = 1, /* attn_decode returns o' (rotated basis); caller folds R_V^T into W_o */
  OSCAR_FLAG_IN_FP32 = 2,  /* k_new, v_new and q are float32 instead of bf16 */
  OSCAR_FLAG_OUT_FP32 = 4, /* attn_decode writes float32 instead of bf16 */
  OSCAR_FLAG_HADAMARD = 8, /* rotate K, V, q and the output by the in-quant Hadamard H (above);
                              R_K and R_V are ignored and may be NULL */
  OSCAR_FLAG_V_BF16 = 16,  /* K-only INT2: V kept BF16 at every position (layout below) */
  OSCAR_FLAG_LLOYD_MAX = 32 /* INT2 codes index Lloyd-Max levels instead of evenly spaced ones (above) */
};

/* return codes */
typedef enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID = -1,     /* null pointer, bad shape, clip not in (0,1], negative window, ... */
  OSCAR_ERR_CAPACITY = -2,    /* n_new or the seq-length hint exceeds capacity */
  OSCAR_ERR_WORKSPACE = -3,   /* workspace smaller than one split needs */
  OSCAR_ERR_LAUNCH = -4,      /* a CUDA launch or attribute call failed */
  OSCAR_ERR_UNSUPPORTED = -5  /* head_dim not in {128, 256, 512}, group != 128, G > 8, or a decode
                                 whose B * Hkv * (S, W or, with OSCAR_FLAG_V_BF16, capacity) >= 2^31 */
} oscar_status;

/* bits OR-ed into *dev_status by the kernels */
enum {
  OSCAR_DEV_OVER_CAPACITY = 1, /* a position or seq_len was >= capacity (row skipped / clamped) */
  OSCAR_DEV_NONFINITE = 2,     /* a non-finite input row */
  OSCAR_DEV_FP16_RANGE = 4,    /* a scale, zero or scaled query component left the fp16 range */
  OSCAR_DEV_TIMEOUT = 8,       /* a pipeline wait gave up (the kernel returned early) */
  OSCAR_DEV_EMPTY = 16,        /* a sequence had seq_len < 1 (its output is zero) */
  OSCAR_DEV_NOT_CONVERGED = 32 /* oscar_calibrate_rk / _rv: Jacobi reached its sweep limit */
};

typedef struct {
  int32_t num_layers;
  int32_t batch;         /* B */
  int32_t num_q_heads;   /* Hq; query head i uses KV head i / (Hq / Hkv) */
  int32_t num_kv_heads;  /* Hkv */
  int32_t head_dim;      /* D: 128, 256 or 512 */
  int32_t group_size;    /* must be 128 */
  int32_t sink;          /* S >= 0: first positions kept BF16 */
  int32_t recent;        /* W >= 0: last positions kept BF16 */
  int32_t capacity;      /* max positions per sequence (> 0) */
  float k_clip;          /* clip ratio for K rows, in (0, 1] */
  float v_clip;          /* clip ratio for V rows, in (0, 1] */
  uint32_t flags;        /* OSCAR_FLAG_* */
} oscar_kv_config;

typedef struct {
  uint64_t ncap;         /* INT2 rows per (sequence, KV head) */
  uint64_t sink_bytes, ring_bytes, codes_bytes, sz_bytes; /* one role of one layer */
  uint64_t role_bytes;   /* K role: sink + ring + codes + sz */
  uint64_t layer_bytes;  /* role_bytes + v_role_bytes (K then V) */
  uint64_t total_bytes;  /* num_layers * layer_bytes */
  uint64_t decode_workspace_bytes; /* attn_decode workspace with OSCAR_KV_MAX_SPLITS slots */
  int32_t max_splits;    /* OSCAR_KV_MAX_SPLITS */
  int32_t reserved;
  uint64_t v_role_bytes; /* V role: role_bytes, or with OSCAR_FLAG_V_BF16 the BF16 rows */
} oscar_kv_layout;

/*
 * kv_layout_query — sizes and offsets of the cache and of the decode
 * workspace.  Host only, pure arithmetic.  Returns OSCAR_ERR_INVALID or
 * OSCAR_ERR_UNSUPPORTED on a bad config, else fills *out.
 * attn_decode with n partial slots needs, with Dg = D/128 and NQT = 2 when
 * Hq/Hkv > 4 else 1,
 *   align256(B*Hkv*Dg*NQT*2048) + align256(B*Hkv*Dg*NQT*4096)
 *   + 2 * align256(B*Hq*Dg*4) + align256(B*Hq*n*D*4) + align256(B*Hq*n*2*4)
 *   + align256(B*Hkv*4) bytes of workspace.
 */
int kv_layout_query(const oscar_kv_config* cfg, oscar_kv_layout* out);

/*
 * kv_append — write n_new new tokens per sequence into layer `layer`.
 *   cache      device, layout above (written).
 *   k_new,v_new device [B][n_new][Hkv][D] post-RoPE rows, bf16 (float32 with
 *              OSCAR_FLAG_IN_FP32).
 *   start_pos  device int32 [B]: position of each sequence's first new token.
 *   R_K, R_V   device float32 [D][D] row-major rotations of this layer
 *              (not read with OSCAR_FLAG_HADAMARD; may then be NULL).
 *   debug_rot_out device float32 [B][n_new][Hkv][2][D] or NULL: receives the
 *              float32 rotated rows the quantiser saw (K then V).
 *   dev_status device int32 or NULL.
 * Position p = start_pos[b] + t gets its INT2 row when p >= S, its sink row
 * when p < S and its ring slot p mod W when p >= start_pos[b] + n_new - W.
 * Rows with p >= capacity are skipped and flagged OSCAR_DEV_OVER_CAPACITY.
 * Enqueued on `stream`; inputs must stay valid until it completes.
 */
int kv_append(const oscar_kv_config* cfg, void* cache, int32_t layer, const void* k_new,
              const void* v_new, const int32_t* start_pos, int32_t n_new, const float* R_K,
              const float* R_V, float* debug_rot_out, int32_t* dev_status, void* stream);

/*
 * attn_decode — one query token per sequence attends to all seq_lens[b]
 * cached positions of layer `layer` (append the current token first).
 *   q          device [B][Hq][D] bf16 (float32 with OSCAR_FLAG_IN_FP32), not rotated.
 *   seq_lens   device int32 [B], 1 <= seq_len <= capacity; a seq_len < 1
 *              gives that sequence a zero output and lse = -inf and sets
 *              OSCAR_DEV_EMPTY, one above capacity is clamped to it and sets
 *              OSCAR_DEV_OVER_CAPACITY.
 *   seq_len_hint host upper bound on seq_lens (0 = capacity); only used to
 *              size the grid when the contexts are short.
 *   R_K, R_V   device float32 [D][D] rotations of this layer (not read
 *              with OSCAR_FLAG_HADAMARD; may then be NULL).
 *   sm_scale   softmax scale; <= 0 means 1/sqrt(D).
 *   num_splits 0 = automatic: one wave of CTAs (as many as are resident at
 *              once).  Else num_splits * B * Hkv CTAs (at most
 *              OSCAR_KV_MAX_SPLITS per unit): with equal seq_lens every
 *              (sequence, KV head) is then split num_splits ways.  Either way
 *              the cache of all (sequence, KV head) units, in unit order, is
 *              cut into equal slices of work, one per CTA, so a CTA can cover
 *              the tail of one unit and the head of the next.
 *   out        device [B][Hq][D] bf16 (float32 with OSCAR_FLAG_OUT_FP32);
 *              o = o' R_V^T, or o' with OSCAR_FLAG_ABSORB_V.  Repeated calls on
 *              the same inputs give the same bits: the CTA that merges a
 *              sequence's KV head (the last of its CTAs to finish) may change
 *              from call to call, but the merge and the un-rotation do the
 *              same arithmetic in the same order in every CTA.
 *   lse        device float32 [B][Hq] or NULL: natural-log log-sum-exp of the
 *              scaled scores.
 *   workspace  device scratch of workspace_bytes (see kv_layout_query); it
 *              holds n = min(OSCAR_KV_MAX_SPLITS, what fits) partial slots per
 *              query head, and no unit is shared by more CTAs than slots (an
 *              explicit num_splits must fit in full).
 * Launches two kernels on `stream`: query rotation (which writes q' as the
 * split kernel's MMA fragments), then split attention whose last CTA per
 * (sequence, KV head) merges that unit's partials and un-rotates V; at
 * head_dim 256 and 512 with V neither absorbed nor Hadamard-rotated a third
 * kernel applies R_V^T to every merged output instead (also at head_dim 128
 * with G > 4 and at most 16 (sequence, KV head) pairs; see
 * oscar_kv_decode_kernels).  All use programmatic
 * dependent launch; the first waits for all prior work on the stream before
 * reading q.  Concurrent calls must not share a workspace.
 */
int attn_decode(const oscar_kv_config* cfg, const void* cache, int32_t layer, const void* q,
                const int32_t* seq_lens, int32_t seq_len_hint, const float* R_K, const float* R_V,
                float sm_scale, int32_t num_splits, void* out, float* lse, void* workspace,
                uint64_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * decode_step — kv_append followed by attn_decode, in one call: the usual
 * decode step of a serving loop (append the current token of every sequence,
 * then attend over the whole context).  Same computation and results as the
 * two calls made in sequence with the same arguments (kv_append of k_new,
 * v_new at start_pos; attn_decode over seq_lens; `out` up to the last bits, as
 * between any two attn_decode calls); the pages' append (Qwen3-4B
 * card, Run; RotationZoo, How to use) and fused attention (hysenlabs article,
 * How the offline rotation is fit) back to back.
 * Because the call knows which cache locations the append writes (the sink
 * positions and INT2 rows of [start_pos[b], start_pos[b] + n_new) and the ring
 * slots of its last min(n_new, W) positions), the attention kernels start
 * streaming every other part of the cache while the append runs, instead of
 * after it.  seq_lens and start_pos must therefore be final when the call is
 * made (they are read before the append completes); q may still be produced
 * by the kernel preceding the call.  Arguments, errors and the workspace are
 * those of kv_append and attn_decode; everything is validated before
 * anything is launched.  Launches the append kernel and attn_decode's kernels
 * on `stream`.
 */
int decode_step(const oscar_kv_config* cfg, void* cache, int32_t layer, const void* k_new, const void* v_new,
                const int32_t* start_pos, int32_t n_new, const void* q, const int32_t* seq_lens,
                int32_t seq_len_hint, const float* R_K, const float* R_V, float sm_scale, int32_t num_splits,
                void* out, float* lse, void* workspace, uint64_t workspace_bytes, int32_t* dev_status,
                void* stream);

/*
 * attn_decode_static — attn_decode for callers that cannot allocate device
 * memory (no counterpart on the pages).  Plugin hosts that own every device
 * allocation, and serving loops that must not call cudaMalloc while other
 * streams run, can call this instead: its scratch is a file-scope __device__
 * array of OSCAR_KV_STATIC_SCRATCH_BYTES inside the library, which every GPU
 * that loads the library holds until the process exits.  Arguments are those of
 * attn_decode without workspace / workspace_bytes; the caller still passes all
 * inputs and outputs.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Returns OSCAR_ERR_WORKSPACE when even one context split needs more
 * scratch than the array holds, or when an explicit num_splits does not fit;
 * the automatic split count is reduced to what fits.  Every call shares the
 * array, so calls whose work overlaps on the GPU race; nothing in it needs to
 * start at zero (each call zeroes its own counters and writes every partial
 * before reading it).
 */
#define OSCAR_KV_STATIC_SCRATCH_BYTES (16u << 20)
int attn_decode_static(const oscar_kv_config* cfg, const void* cache, int32_t layer, const void* q,
                       const int32_t* seq_lens, int32_t seq_len_hint, const float* R_K, const float* R_V,
                       float sm_scale, int32_t num_splits, void* out, float* lse, int32_t* dev_status,
                       void* stream);

/*
 * oscar_kv_set_profile_events — measurement hook (no counterpart on the pages).
 * While both events are non-NULL (cudaEvent_t passed as void*), every
 * attn_decode call made from the calling host thread records `split_start` on
 * its stream immediately before launching the split-attention kernel and
 * `split_stop` immediately after it and the un-rotation kernel that may
 * follow it (see oscar_kv_decode_kernels), so that cudaEventElapsedTime gives
 * the device time of the attention proper.  Recording between kernels removes the launch overlap
 * of that call.  Pass NULL, NULL to stop.  The setting is per host thread.
 */
int oscar_kv_set_profile_events(void* split_start, void* split_stop);

/*
 * oscar_kv_decode_kernels — how many kernels one attn_decode call with this
 * configuration launches (no counterpart on the pages; for launch accounting
 * and graph planning): query rotation and split attention, plus an
 * un-rotation kernel when V is neither absorbed nor Hadamard-rotated and
 * either head_dim is 256 / 512 or more than four query heads share a KV head
 * with at most 16 (sequence, KV head) pairs in the batch.  decode_step launches one kernel more (the append).
 * Needs no device.  Returns 2 or 3, or OSCAR_ERR_INVALID for an invalid
 * configuration.
 */
int oscar_kv_decode_kernels(const oscar_kv_config* cfg);

/*
 * oscar_kv_set_wait_test — test hook for the device-timeout path (no
 * counterpart on the pages).  Every wait of the split-attention kernel on one
 * of its shared-memory barriers is bounded; when the bound runs out the kernel
 * ORs OSCAR_DEV_TIMEOUT into *dev_status, waits (bounded again) for the copies
 * it issued, skips the rest of its work and returns, leaving the context
 * usable.  For attn_decode / decode_step calls made later from the calling host
 * thread this hook sets that bound to wait_ns (0 = the default, about 2 s) and
 * makes the first copy issued by CTA 0 expect `extra_bytes` more than its copies
 * deliver, so that its barrier never completes and the bounded wait runs out;
 * every copy still completes.  (0, 0) restores normal operation.  A decode run
 * with extra_bytes > 0 leaves at least one output unit unwritten.  Returns
 * OSCAR_ERR_INVALID for wait_ns > 10 s or extra_bytes outside [0, 2^20].
 */
int oscar_kv_set_wait_test(uint64_t wait_ns, int32_t extra_bytes);

/*
 * oscar_calibrate_rk — the K-side rotation fitted to a calibration set of
 * query rows ["OSCAR-RotationZoo" card, File format: R_K = R H P_br with R the
 * eigenvectors of the query covariance, H a head-dim Hadamard and P_br the
 * eigenvalue-sorted bit-reversal permutation; hysenlabs article, How the
 * offline rotation is fit: activations captured offline, rotation derived
 * from their covariance].  Offline work, not part of the decode path.
 *   q          device [n_rows][head_dim] float32 query rows of one layer
 *              (post-RoPE; every head's rows pooled), 16-byte aligned.
 *   n_rows     1 .. OSCAR_KV_CALIB_MAX_ROWS.
 *   R_K_out    device [head_dim][head_dim] float32, row-major, written:
 *              Sigma = q^T q in float64; E = its eigenvectors (one-sided
 *              Jacobi in float64 on a cooperative grid) ordered by descending
 *              eigenvalue (ties by index),
 *              each column signed so that its largest-magnitude entry (the
 *              first, on ties) is positive; R_K = E H P_br with
 *              H[i][k] = (-1)^popcount(i & k) / sqrt(D) and column j of R_K
 *              = column br(j) of E H (br reverses the log2 D bits of j).
 *   workspace  device, >= the size oscar_calibrate_workspace_query returns,
 *              256-byte aligned; caller owned, contents undefined after.
 * Launches three kernels on `stream` (the second as a cooperative launch).
 * A Jacobi that reaches its sweep limit (40 sweeps) sets OSCAR_DEV_NOT_CONVERGED in *dev_status; the result is
 * then the last iterate.  Errors: OSCAR_ERR_INVALID (null or misaligned
 * pointer, n_rows out of range), OSCAR_ERR_UNSUPPORTED (head_dim),
 * OSCAR_ERR_WORKSPACE, OSCAR_ERR_LAUNCH.
 */
int oscar_calibrate_workspace_query(int32_t head_dim, uint64_t* bytes);
int oscar_calibrate_rk(const float* q, int64_t n_rows, int32_t head_dim, float* R_K_out, void* workspace,
                       uint64_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * oscar_calibrate_rv — the V-side rotation fitted to the score-weighted V
 * covariance ["OSCAR-RotationZoo" card, File format: the V rotation is built
 * on V^T diag(K^T (Q^T Q) K) V with the same R H P_br construction].  The
 * printed product composes when K holds the keys as columns: K^T Q^T Q K is
 * then S^T S for the logits S of every calibration query against every key,
 * and its diagonal is each key's score energy.  Offline work.
 *   q          device [n_q_rows][head_dim] float32 query rows of one layer
 *              (post-RoPE, every head's rows pooled), 16-byte aligned.
 *   k, v       device [n_kv_rows][head_dim] float32 key and value rows of the
 *              same layer (row t of k and of v: one token of one KV head),
 *              16-byte aligned.
 *   n_q_rows, n_kv_rows  1 .. OSCAR_KV_CALIB_MAX_ROWS.
 *   R_V_out    device [head_dim][head_dim] float32, row-major, written:
 *              Sigma_Q = q^T q and w_t = k_t Sigma_Q k_t^T in float64,
 *              Sigma_V = sum_t w_t v_t^T v_t in float64, then E, its sign
 *              convention, H and P_br exactly as oscar_calibrate_rk does for
 *              Sigma.
 *   workspace  device, >= the size oscar_calibrate_rv_workspace_query returns
 *              (it grows with n_kv_rows), 256-byte aligned; caller owned,
 *              contents undefined after.
 * Launches five kernels on `stream` (the fourth as a cooperative launch) and
 * two memsets.  Sweep
 * limit, status bits and errors as oscar_calibrate_rk.
 */
int oscar_calibrate_rv_workspace_query(int32_t head_dim, int64_t n_kv_rows, uint64_t* bytes);
int oscar_calibrate_rv(const float* q, int64_t n_q_rows, const float* k, const float* v, int64_t n_kv_rows,
                       int32_t head_dim, float* R_V_out, void* workspace, uint64_t workspace_bytes,
                       int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_KV_H */
