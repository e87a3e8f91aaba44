/*
 * lean_attn.h -- C ABI of the LeanAttention decode-phase attention library
 * (stream-K decode attention for one GPU, sm_103a).
 *
 * The operation (xllm-io paper review of LeanAttention, "3.1 standard
 * attention", decode phase with one query token): for every request b and
 * query head h,
 *     s_t   = scale * q[b,h,:] . K[b, h/grp, t, :]      t < L_b
 *     out[b,h,:] = sum_t softmax(s)_t V[b, h/grp, t, :]
 * with grp = hq / hkv query heads sharing one kv head.
 *
 * How it is computed (same review, "3.3 LeanTile" to "3.5 execution flow",
 * and "3.2 softmax rescaling as a reduction"): the context of every
 * (request, kv head) unit is cut into LeanTiles (256 tokens at d = 64, 128
 * tokens at d = 128); all tiles are laid out on one line and split evenly
 * over G CTAs, which may cross head and request boundaries; each CTA
 * produces partial results (m, l, unscaled O) that the unit's host CTA
 * merges with the rescaling reduction f and normalises, all in one launch
 * (for units of more than 16 query rows, and for units of 4-16 rows whose
 * host would read at least 96 KiB of records, every CTA that ends on a
 * piece of the unit merges an equal share of its outputs instead).
 *
 * Data layout (device memory, row-major, no padding):
 *   q    [batch, hq, d]                         fp16 or bf16
 *   k, v request b is a contiguous [hkv, L_b, d] slab starting at element
 *        hkv * cu[b] * d; token t of kv head h sits at element
 *        (hkv * cu[b] + h * L_b + t) * d.  With equal lengths this is the
 *        [batch, heads, seq_len, head_dim] layout the review's "7.4
 *        limitations" names.                    fp16 or bf16 (same as q)
 *   cu_seqlens_k  int32 [batch + 1], cu[0] = 0, cu[b+1] - cu[b] = L_b >= 1
 *   out  [batch, hq, d]                         fp32
 *
 * Threading and ownership: the caller owns every buffer and the stream.
 * A schedule is owned by the library until la_schedule_destroy; it keeps a
 * device copy of its tables, uploaded on its first la_decode (that call
 * allocates device memory and synchronises, so make it before any stream
 * capture). A schedule may be used from one thread at a time.
 *
 * Errors: every entry point returns an la_status and never throws. Argument,
 * shape and support problems are reported before anything is launched.
 * la_decode is asynchronous; a failure detected inside the kernel (a
 * bounded wait that ran out, a cu_seqlens_k that disagrees with the
 * schedule) is recorded in the workspace and returned by la_get_status.
 */
#ifndef LEAN_ATTN_H
#define LEAN_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* la_stream_t;

typedef struct la_schedule la_schedule;

typedef enum {
  LA_OK = 0,
  LA_ERR_INVALID = 1,     /* bad argument, shape, pointer or alignment */
  LA_ERR_UNSUPPORTED = 2, /* a valid shape this build does not implement */
  LA_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  LA_ERR_TIMEOUT = 4,     /* a bounded wait inside the kernel ran out */
  LA_ERR_WORKSPACE = 5    /* workspace missing, too small or misaligned */
} la_status;

typedef enum { LA_F16 = 0, LA_BF16 = 1 } la_dtype;

/* Element type of the output of la_decode_ex. */
typedef enum { LA_OUT_F32 = 0, LA_OUT_F16 = 1, LA_OUT_BF16 = 2 } la_dtype_out;

/* Kinds of work a CTA does on one unit, as exported by la_schedule_export. */
enum {
  LA_SEG_WHOLE = 0,   /* the CTA covers the whole unit: normalise, write out */
  LA_SEG_NONHOST = 1, /* a later piece: write (m, l, O) to the workspace, set a ready flag */
  LA_SEG_HOST = 2,    /* the first piece: wait for the later pieces, merge with f, write out */
  LA_SEG_PARTIAL = 3  /* fixed-split piece: write (m, l, O); a second launch merges */
};

/*
 * la_plan -- the stream-K tile planner ("3.4 stream-K style decomposition"
 * and "3.5 execution flow" of the xllm-io review).
 *
 *   batch, hq, hkv, d  shape; d in {64, 80, 96, 128, 256}; hq % hkv == 0
 *                      (any group grp = hq / hkv). Up to 16 query rows per
 *                      kv head run as one unit on the 16-row kernel; a group
 *                      that is not a power of two runs on the next larger
 *                      instance (1, 2, 4, 8 or 16 rows), whose spare rows are
 *                      zero queries never written out. A unit of 17-128
 *                      rows (17-64 at d = 256; e.g. multi-query attention)
 *                      runs on the tcgen05 kernel (128-lane instance,
 *                      128-token tiles, 64 at d = 256). A kv head with more
 *                      rows than a unit holds (128; 64 at d = 256) is split into
 *                      query blocks: the fewest equal blocks of consecutive
 *                      query heads that fit (qb blocks of grp / qb heads, qb
 *                      dividing grp); every block is a unit of its own that
 *                      reads the kv head's K/V
 *   cu_seqlens_k       HOST pointer to batch + 1 int32 offsets (read, not kept)
 *   num_sms            grid size G; <= 0 picks one persistent CTA per SM of
 *                      the current device (the kernel runs one CTA per SM).
 *                      A G larger than the device can hold at once is
 *                      rejected by la_decode, because host CTAs wait for
 *                      later CTAs inside the launch.
 *   out                receives the new schedule
 *
 * Rules: tiles(b) = ceil(L_b / T) with the default T of la_plan_ex
 * (the review's table: 256 at d = 64, 128 at d = 128; 64 at d = 128 with
 * one or two query heads per kv head, measured faster on GB300);
 * units (b, kv head[, query block]) in request-major order, then kv head,
 * then query block; I = total tiles; CTA g takes
 * floor(I/G) iterations plus one if g < I mod G, in order; the host of a
 * unit is the CTA holding its first tile, the finisher the one holding its
 * last. Pure host code when num_sms > 0. Returns LA_ERR_INVALID for bad
 * shapes or lengths, LA_ERR_UNSUPPORTED for d or group sizes not built.
 */
la_status la_plan(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k, int num_sms,
                  la_schedule** out);

/*
 * la_plan_ex -- la_plan with more head dims and a chosen LeanTile size (the
 * review's "7.4 limitations": the best LeanTile depends on the hardware and
 * the configuration, so it is a parameter).
 *
 *   d            64, 80, 96, 128 or 256
 *   tile_tokens  0 for the default of d, else one of the built sizes:
 *                d = 64: 256 (default) or 128;  d = 128: 128 or 64;
 *                d = 80, 96: 128;  d = 256: 64.
 *                The table gives 256 and 128 tokens for d = 64 and 128
 *                (64 KiB of K+V per tile); the other defaults keep a tile
 *                near that size (40, 48 and 64 KiB). At d = 128 the default
 *                is 64 when a unit has at most 2 query rows (group x query
 *                tokens; the CUDA-core tile path): on GB300 the smaller
 *                tile measured 1.1-1.3 % faster on uniform, ragged and
 *                512k-context batches; with 4-8 rows (tensor-core path)
 *                the table's 128 stays faster (2-3 %), and so it does for
 *                la_plan_fixed, whose few busy SMs each need the deeper
 *                shared-memory ring of the larger tile. Units of more
 *                than 16 query rows (the tcgen05 kernel) take 128 only
 *                (64 at d = 256).
 * Other arguments and rules as la_plan. LA_ERR_UNSUPPORTED for a (d, T)
 * that is not built.
 */
la_status la_plan_ex(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k, int num_sms,
                     int tile_tokens, la_schedule** out);

/*
 * la_plan_spec -- stream-K schedule for nq query tokens per request, as in
 * speculative-decoding verification (the review's "7.4" lists combining
 * the method with speculative decoding as future work).
 *
 * The nq query tokens of request b are the last nq tokens of its context:
 * query i (0 <= i < nq) sits at position L_b - nq + i and attends to keys
 * 0 .. L_b - nq + i (a causal mask inside the last tile). With such a
 * schedule la_decode / la_decode_ex / la_decode_kv / la_decode_static read
 * q as [batch, nq, hq, d] and write out as [batch, nq, hq, d]. The tiles and
 * their split are those of la_plan (K/V are read once per kv head for all
 * grp * nq query rows, as many as a unit holds; above that the kv head's
 * query heads are split into query blocks as in la_plan, each of
 * grp / qb * nq rows). Requires nq <= 128 (64 at d = 256;
 * LA_ERR_UNSUPPORTED), and L_b >= nq for every request
 * (LA_ERR_INVALID); nq = 1 is la_plan.
 */
la_status la_plan_spec(int batch, int hq, int hkv, int d, int nq, const int32_t* cu_seqlens_k, int num_sms,
                       la_schedule** out);

/*
 * la_plan_fixed -- fixed partitions used as baselines (the review's "2.2"
 * and "2.3" on FlashAttention-2 and FlashDecoding, and "4.3" on their
 * relation to the stream-K mapping). Every unit is cut into
 * min(splits, tiles) even pieces, one CTA each. splits == 1: one CTA per
 * (request, kv head), no reduction. splits > 1: every piece writes its
 * partial result and a second kernel merges them (two launches per call).
 * No CTA waits on another, so G is not limited by co-residency.
 */
la_status la_plan_fixed(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k,
                        int splits, la_schedule** out);

/*
 * la_plan_auto -- shape-driven choice among the three partitions (the
 * Silicon & Systems digest's "a useful control policy": a runtime picks a
 * FlashAttention-style, fixed-split or stream-K schedule from the shape;
 * the xllm-io review's "4.3" shows the first two are special cases).
 *
 * Builds the stream-K schedule over num_sms CTAs (<= 0: one per SM of the
 * current device), the one-CTA-per-unit partition and the fixed split into
 * max(2, ceil(SMs / units)) pieces, predicts each one's time and returns
 * the fastest. Time model: CTAs dispatched in order onto the SMs as they
 * free up; n running CTAs read 7.5 TB/s * (1 - exp(-n / 60)) together
 * (fitted to GB300 measurements); 3 us of start-up per CTA an SM runs in
 * turn, 2.5 us for host CTAs' merges (for units of more than 16 rows,
 * 3 us + 0.11 us per piece of a unit), 8 us per launch and 4 us for the
 * second (merge) launch of a fixed split (+ 0.13 us per piece of a unit
 * above 16 rows).
 * predicted_us: NULL, or 3 doubles receiving the predictions (stream-K,
 * one per unit, fixed split). The returned schedule is used like any
 * other; la_schedule_export tells which kind it is (word 6, word 7).
 */
la_status la_plan_auto(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k, int num_sms,
                       la_schedule** out, double* predicted_us);

/* Grid size G of a schedule (CTAs per launch), or -1 for NULL. */
int la_schedule_grid(const la_schedule* s);

/*
 * Bytes of device workspace la_decode needs for this schedule: a 256-byte
 * header, ready flags (padded to 256 bytes) and partial records, one flag
 * per record ("7.4 limitations": a small amount of global memory for
 * sharing partial results). The 16-row kernel has records of rows rows of
 * [m, l, 0, 0, O[d]] floats (rows = query rows per unit head -- a kv head
 * or one query block of one -- rounded up to 1, 2, 4, 8 or 16, times the kv
 * heads per unit): G of them below 4 rows, 2 G from 4 rows (a unit split
 * into many pieces is then merged by every CTA that ends on one of them, so
 * each piece writes a record and a CTA can hold two); the tcgen05 kernel
 * (128 rows) 2 G records of the same triples column-major over the rows,
 * rounded up to a multiple of 4 floats. Zero it
 * once (la_workspace_init) before its first use; after that it needs no
 * clearing between calls. One workspace must not be used by two launches
 * that can run at the same time.
 */
size_t la_workspace_size(const la_schedule* s);

/* Zero a workspace on a stream (cudaMemsetAsync). */
la_status la_workspace_init(void* workspace, size_t bytes, la_stream_t stream);

/*
 * la_decode -- one decode-attention call, enqueued on `stream`.
 *
 *   q, k, v           device pointers, layout above, 16-byte aligned
 *   dt                element type of q, k and v
 *   cu_seqlens_k_dev  DEVICE copy of the offsets the schedule was planned
 *                     with; the kernel checks it against the schedule and
 *                     reports LA_ERR_INVALID through la_get_status if they
 *                     differ (the affected outputs are NaN)
 *   s                 schedule from la_plan or la_plan_fixed
 *   workspace         device memory of la_workspace_size(s) bytes,
 *                     256-byte aligned, zeroed once before first use
 *   out               device fp32 [batch, hq, d], 16-byte aligned
 *   scale             multiplies every score before the softmax (1/sqrt(d)
 *                     in the review's formula)
 *
 * One kernel launch for stream-K schedules (plus one merge launch for
 * fixed splits > 1). Does not synchronise, except on a schedule's first
 * use (upload of its tables). Kernels are launched as programmatic
 * dependents (cudaLaunchAttributeProgrammaticStreamSerialization): their
 * CTAs may be placed while the kernel before them on the stream finishes,
 * but each first waits (griddepcontrol.wait) until that kernel has
 * completed and its writes are visible, so stream order is kept for every
 * byte read or written. Returns LA_ERR_INVALID / LA_ERR_WORKSPACE for bad
 * arguments, LA_ERR_CUDA if a launch fails.
 */
la_status la_decode(const void* q, const void* k, const void* v, la_dtype dt,
                    const int32_t* cu_seqlens_k_dev, const la_schedule* s, void* workspace,
                    float* out, float scale, la_stream_t stream);

/*
 * la_decode_ex -- la_decode with a choice of output element type: out is
 * [batch, hq, d] of fp32 (LA_OUT_F32, what la_decode writes), fp16 or bf16
 * (rounded to nearest even from the fp32 result); 16-byte aligned.
 * LA_ERR_INVALID for an unknown out_dt; otherwise as la_decode.
 */
la_status la_decode_ex(const void* q, const void* k, const void* v, la_dtype dt,
                       const int32_t* cu_seqlens_k_dev, const la_schedule* s, void* workspace,
                       void* out, la_dtype_out out_dt, float scale, la_stream_t stream);

/*
 * K/V cache layouts for la_decode_kv (the review's "7.4 limitations" notes
 * that the method asks for a [batch, heads, seq_len, head_dim] layout;
 * serving stacks keep a token-major or paged cache instead).
 *   LA_KV_SLAB         request b is a [hkv, L_b, d] slab at element
 *                      hkv*cu[b]*d (the layout of la_decode)
 *   LA_KV_TOKEN_MAJOR  [total tokens, hkv, d]: token t of request b, kv
 *                      head h at element ((cu[b] + t)*hkv + h)*d
 *   LA_KV_PAGED        [num_pages, page_size, hkv, d]: token t of request b
 *                      sits in page block_table[b*max_blocks + t/page_size]
 *                      at slot t % page_size
 * Both non-slab layouts are read with 3-D TMA loads; page ids outside
 * [0, num_pages) read as zeros, never out of bounds.
 */
typedef enum { LA_KV_SLAB = 0, LA_KV_TOKEN_MAJOR = 1, LA_KV_PAGED = 2 } la_kv_layout;

typedef struct {
  la_kv_layout layout;
  const int32_t* block_table; /* paged: DEVICE int32 [batch, max_blocks] page ids */
  int max_blocks;             /* paged: row stride of block_table, >= ceil(max L_b / page_size) */
  int page_size;              /* paged: tokens per page, a power of two >= 16 */
  long long num_pages;        /* paged: pages in each of the K and V caches */
} la_kv_desc;

/*
 * la_decode_kv -- la_decode_ex on a cache in any of the layouts above
 * (k and v point at the caches; cu_seqlens_k_dev still gives the context
 * lengths). LA_ERR_INVALID for a bad descriptor (page size not a power of
 * two >= 16, too few block-table columns, NULL table); LA_ERR_UNSUPPORTED
 * when a page is too small for the tensor-core path's swizzled pieces
 * (d = 80 with groups 4/8 needs page_size >= 32) or the cache has more than
 * 2^31 - 1 token rows.
 */
la_status la_decode_kv(const void* q, const void* k, const void* v, la_dtype dt,
                       const int32_t* cu_seqlens_k_dev, const la_kv_desc* kv, const la_schedule* s,
                       void* workspace, void* out, la_dtype_out out_dt, float scale, la_stream_t stream);

/*
 * la_plan_kv -- stream-K schedule for a token-major or paged cache whose
 * rows of one kv head are short (d * 2 bytes < 256, i.e. d = 64, 80, 96).
 * The paper has no counterpart: its units are single (request, head) pairs
 * over a [batch, heads, seq_len, head_dim] layout. In a token-major or paged
 * cache the d elements of one kv head are only 128-192 contiguous bytes of
 * each token row; read one head at a time they stream at 0.5-0.85 of the
 * copy rate on GB300. A unit of several kv heads reads those heads of every
 * token row together, in whole 256-byte multiples where it can (d = 64: two
 * heads, 256 bytes; d = 96: four, 768 bytes; d = 80: eight, 1280 bytes).
 *
 *   nq              query tokens per request, as la_plan_spec (1: decode)
 *   heads_per_unit  kv heads of one unit. Built: 1 (any d); d = 64: 2;
 *                   d = 80: 2, 8; d = 96: 2, 4 (up to 8 query rows per kv
 *                   head; more rows need 1). 0 picks the fewest heads
 *                   whose rows make whole 256-byte pieces if that count
 *                   divides hkv, else the most built count that divides
 *                   hkv, else 1 (always 1 for d = 128, 256, for more
 *                   than 8 query rows per kv head and for query blocks).
 *   tile_tokens     tokens of each head per tile; 0 picks the default:
 *                   the review's table size of d (128 at d = 128 also for
 *                   one or two query rows: 16-token pages read 13 % slower
 *                   with 64) divided by heads_per_unit, so a tile still
 *                   holds the same bytes (only these defaults are built for
 *                   more than one head per unit); 128 (64 at d = 256) for
 *                   units of more than 16 query rows (the tcgen05 kernel).
 *   num_sms, out    as la_plan
 * Units are (request, group of heads_per_unit consecutive kv heads) in
 * request-major order, tiles(b) = ceil(L_b / tile_tokens), and the split
 * rules are la_plan's over hkv / heads_per_unit heads. A schedule with more
 * than one head per unit runs with la_decode_kv on LA_KV_TOKEN_MAJOR or
 * LA_KV_PAGED caches only (la_decode, la_decode_ex, la_decode_static and
 * the slab layout return LA_ERR_UNSUPPORTED); its la_schedule_export
 * counts units of heads_per_unit heads. LA_ERR_INVALID when heads_per_unit
 * is not 0, 1, 2, 4 or 8 or does not divide hkv; LA_ERR_UNSUPPORTED for a
 * count or tile that is not built; otherwise the errors of la_plan_spec.
 */
la_status la_plan_kv(int batch, int hq, int hkv, int d, int nq, const int32_t* cu_seqlens_k,
                     int heads_per_unit, int tile_tokens, int num_sms, la_schedule** out);

/*
 * la_decode_static -- la_decode without a workspace and without any device
 * allocation. The paper has no counterpart: this is a library convenience.
 *
 * Some callers cannot allocate device memory: a plugin loaded into a host
 * program whose allocator it cannot reach, or a serving loop that reserves
 * all of HBM for its KV cache up front and must not call cudaMalloc (which
 * can synchronise the device) while it decodes. This call keeps the
 * kernel's scratch (ready flags, partial records and the schedule's
 * tables) in one fixed 4 MiB array of device memory built into the
 * library; every GPU that loads the library holds that array until the
 * process exits. Arguments are those of la_decode minus the workspace.
 *
 *   - A schedule whose scratch does not fit in 4 MiB is rejected with
 *     LA_ERR_WORKSPACE before anything is enqueued (about 7,000 CTA records
 *     at d = 128 without query-head grouping; use la_decode for more).
 *     Where the second record per CTA of the shared merge (see
 *     la_workspace_size) does not fit but one does, every split unit is
 *     merged at its host instead.
 *   - The first call on a device looks up the array's address on that
 *     device (cudaGetSymbolAddress) with the device current; make that
 *     first call before any stream capture.
 *   - Each call clears the array's header and ready flags on `stream`,
 *     then launches the same kernel(s) as la_decode. The schedule's tables
 *     are copied from host memory into the array only when the array on
 *     this device does not already hold them (the first call with a
 *     schedule, or a call after one with another schedule); a run of calls
 *     with one schedule copies them once. All calls share the one array,
 *     which keeps the previous call's contents: calls that can overlap on
 *     the GPU (on different streams, or from several threads) race, so
 *     serialise them.
 *   - There is no status word to read back: a failure detected inside the
 *     kernel shows up as NaN outputs.
 */
la_status la_decode_static(const void* q, const void* k, const void* v, la_dtype dt,
                           const int32_t* cu_seqlens_k_dev, const la_schedule* s, float* out,
                           float scale, la_stream_t stream);

/*
 * la_decode_host -- one decode call on inputs in HOST memory, with the copies
 * in and out enqueued on `stream` around it (the paper has no counterpart:
 * its measurements start with q, K and V already on the device). On
 * `stream`, in order: q_host -> q_dev, k_host -> k_dev, v_host -> v_dev
 * (one cudaMemcpyAsync each), la_decode on the device copies, then
 * out_dev -> out_host. Sizes follow the schedule: q and out hold
 * batch * nq * hq * d elements (fp16/bf16 and fp32), k and v
 * hkv * cu[batch] * d elements each, in la_decode's slab layout.
 *
 *   q_host, k_host, v_host, out_host  host buffers; page-locked memory
 *                     (cudaHostAlloc / cudaHostRegister) makes the copies
 *                     asynchronous. Read q/k/v and write out_host only
 *                     after the stream has reached this call's end.
 *   q_dev, k_dev, v_dev, out_dev      device buffers of those sizes,
 *                     16-byte aligned, owned by the caller
 *   other arguments   as la_decode
 * Does not synchronise (except on a schedule's first use, as la_decode).
 * The arguments are checked before anything is enqueued: LA_ERR_INVALID /
 * LA_ERR_WORKSPACE as la_decode, LA_ERR_UNSUPPORTED for schedules of
 * several kv heads per unit, LA_ERR_CUDA if a copy or launch fails.
 */
la_status la_decode_host(const void* q_host, const void* k_host, const void* v_host, la_dtype dt,
                         const int32_t* cu_seqlens_k_dev, const la_schedule* s, void* q_dev, void* k_dev,
                         void* v_dev, void* workspace, float* out_dev, float* out_host, float scale,
                         la_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the first error a kernel
 * recorded in `workspace` since the last call (LA_OK if none). Meant for
 * tests and error handling, not for the hot loop.
 */
la_status la_get_status(void* workspace, la_stream_t stream);

/*
 * Planner parity: the schedule as int32 words,
 *   [0x4C41, G, U, I, T, nseg, kind (0 stream-K, 1 fixed), splits]
 *   cta_iter[G+1]  first global tile iteration of every CTA (+ total)
 *   unit_iter[U+1] first global tile iteration of every unit (+ total)
 *   cta_seg[G+1]   first segment of every CTA (+ total)
 *   segs[nseg*5]   (unit, tile_begin, tile_end, LA_SEG_* kind, peer): peer
 *                  is the finishing CTA for LA_SEG_HOST, else -1
 *   unit_host[U], unit_fin[U]
 * la_schedule_export_size gives the word count; la_schedule_export fails
 * with LA_ERR_INVALID if n is smaller.
 */
size_t la_schedule_export_size(const la_schedule* s);
la_status la_schedule_export(const la_schedule* s, int32_t* buf, size_t n);

/*
 * Test hooks for failure detection (no GPU fault is ever needed):
 *   skip_signal_cta  CTA that never sets the ready flag of its first segment
 *                    (-1: none), so the bounded waits of the CTAs merging that
 *                    segment's unit run out and report LA_ERR_TIMEOUT
 *   spin_timeout_ns  limit of every wait inside the kernel (default 2 s)
 */
la_status la_schedule_set_debug(la_schedule* s, int skip_signal_cta, long long spin_timeout_ns);

/*
 * Depth of the shared-memory ring the decode kernel cycles through (a
 * tuning knob; the paper has no counterpart). Each CTA holds 2-4 stages of
 * one LeanTile of K plus one of V within 192 KiB; stages = 0 restores the
 * library's choice, 2-4 requests that many (capped at what the kernel
 * instance holds). The library's choice: every stage for the fixed
 * partitions, whose few busy SMs each need many bytes in flight; for
 * stream-K over every SM, 3 stages at d = 96 and 2 at d = 128 with
 * 128-token tiles (slab and paged layouts), where fewer bytes in flight
 * per SM measured faster on GB300. Results do not depend on it (every warp
 * sees the same tokens in the same order). LA_ERR_INVALID for other values.
 */
la_status la_schedule_set_stages(la_schedule* s, int stages);

/*
 * Optional per-CTA timeline, to measure the balance of work across SMs and
 * how long host CTAs wait for partial results (the talk's "temporal skew").
 * trace_dev: device buffer of la_schedule_grid(s) * 8 uint64 words (8-byte
 * aligned), or NULL to stop tracing. Per CTA, in globaltimer nanoseconds
 * unless noted: [0] SM id, [1] kernel entry, [2] first tile landed,
 * [3] last tile consumed, [4] total host wait (ns), [5] end,
 * [6] tiles processed, [7] segments processed. The buffer is written by
 * every later la_decode with this schedule until tracing is turned off.
 */
la_status la_schedule_set_trace(la_schedule* s, void* trace_dev);

/* Most CTAs of the stream-K kernel one SM of the current device holds for
 * head dim d and group size grp (any grp >= 1; above 16, the instance of its
 * query blocks), and the SM count. */
la_status la_device_capacity(int d, int grp, int* ctas_per_sm, int* num_sms);

void la_schedule_destroy(la_schedule* s);

const char* la_status_string(la_status st);

#ifdef __cplusplus
}
#endif

#endif /* LEAN_ATTN_H */
