/*
 * attn.h -- C-ABI of libattn.so, a GB300 (sm_103a) fused attention forward.
 *
 * The operation.  For every batch b, query head hq and query row i:
 *
 *     O[b,hq,i,:] = sum_j softmax_j( scale * <Q[b,hq,i,:], K[b,hkv,j,:]> + mask(i,j) ) V[b,hkv,j,:]
 *     LSE[b,hq,i] = ln sum_{kept j} exp( scale * <Q[b,hq,i,:], K[b,hkv,j,:]> )
 *
 * with hkv = hq / (Hq / Hkv) (grouped-query attention: contiguous groups of
 * query heads share one key/value head), computed tile by tile with a running
 * max and running sum so the S x S score matrix never reaches memory.  This is
 * the FlashAttention scheme the page "NVIDIA让AI狂肝7天自己写算子"
 * (yetianai.com/news/16520) describes in its FlashAttention-lineage section
 * (block-wise computation that never stores the full attention matrix); the
 * masks and the score scaling follow the page "Opus 4.6 + AutoResearch驱动25轮
 * 迭代..." (yunpan.plus/t/19526-1-1), code excerpt "Apply mask + scale
 * in-register"; causal and non-causal prefill and GQA are the workloads of the
 * benchmark section of the first page named above.
 *
 * mask(i,j) is 0 for a kept entry and -inf for a masked one.  Entry (i,j) is
 * kept when (causal == 0 || j <= i) and (mask_bits == NULL || bit j%32 of word
 * mask_bits[b][i][j/32] is 1).  A row with no kept entry is defined as O = 0
 * and LSE = -inf.
 *
 * Conventions for every entry point:
 *   - q, o:   [B][Hq][S][d] row-major, contiguous, device memory, 16-byte aligned.
 *   - k, v:   [B][Hkv][S][d] row-major, contiguous, device memory, 16-byte aligned.
 *   - lse:    float [B][Hq][S], device memory, natural log; may be NULL (not written).
 *   - mask_bits: uint32 [B][S][ceil(S/32)], device memory, 4-byte aligned, least-
 *             significant bit first, 1 = attend, shared by all heads of a batch
 *             entry; bits past column S-1 are ignored.  NULL = no custom mask.
 *   - d in {64, 128}; Hq % Hkv == 0; B, Hq, Hkv, S >= 1; scale > 0 and finite.
 *   - dtype: ATTN_F16 or ATTN_BF16 (q, k, v and o share it); accumulation is fp32.
 *   - stream: a cudaStream_t (NULL = the legacy default stream).
 *   - Ownership: the caller owns every buffer; the library keeps no pointer to
 *     them after the call returns.  The library's own state is small and cached:
 *     tensor maps (TMA descriptors) keyed by buffer address, shape and tile box,
 *     reused by later calls on the same buffers (a map holds only these, so a
 *     cached one stays valid); a status word per (device, stream); and, per
 *     (device, stream) that has run a custom mask, one workspace.  Without a
 *     custom mask nothing is allocated.  With one, a pre-pass kernel writes the
 *     kept-bit words (mask AND causal AND the key bound, padded to whole
 *     128-column tiles; when no bound applies, the key count is a multiple of
 *     128 and mask_bits is 16-byte aligned those equal mask_bits, which the
 *     attention kernel then reads in place) and an emptiness map per (16-row
 *     block, 128-column tile),
 *     and a compaction kernel lists, per mask row block, the 16-row blocks that
 *     keep anything: the attention kernel computes only those, packed eight to a
 *     128-row tile, and writes O = 0, LSE = -inf for the rows of the others
 *     without computing them.  That output lives in the stream's workspace, of at
 *     least the "custom-mask scratch size": with nm mask row blocks (B, or B*Hq
 *     for per-head masks), R = ceil(Sq/16), T = ceil(Sq/128), U = ceil(Sq/256)
 *     and N = ceil(Sk/128), the sum of nm*Sq*N*16, nm*R*N, nm*R, nm*U*64 and
 *     nm*T*N bytes, each rounded up to a multiple of 256 (Sq = Sk = S for
 *     attn_fwd).  The workspace is a stream-ordered allocation (cudaMallocAsync
 *     on `stream`, whole MiB) made by the first custom-mask call on the stream
 *     and reused by every later one; a call that needs more frees the old block
 *     in stream order (cudaFreeAsync) and allocates a larger one.  Repeated calls
 *     of one shape therefore allocate nothing after the first.  Variable-length
 *     batches (attn_fwd_ex with per-entry lengths or packed offsets) use the same
 *     workspace for their work order, B*ceil(max Sq/256) ints after the mask
 *     scratch (256-byte aligned).  The workspace is held until
 *     attn_release_workspace(stream) or process exit: release it before
 *     destroying a stream that has run custom masks or variable-length batches.
 *   - Errors: arguments are validated before any launch (ATTN_ERR_INVALID /
 *     ATTN_ERR_UNSUPPORTED, nothing launched); a failed launch returns
 *     ATTN_ERR_CUDA.  The work is asynchronous: a kernel that gives up on a
 *     barrier wait (see attn_set_wait_timeout_ns) records ATTN_ERR_TIMEOUT in
 *     the status word of the stream it was launched on, which attn_check(that
 *     stream) reports.  The library never traps and never exits the process.
 *   - Thread safety: calls on different streams may run concurrently, and so may
 *     host threads calling on one stream (the library's caches are guarded by
 *     mutexes), except attn_fwd_noalloc with a custom mask: its calls share one
 *     fixed array and must not overlap on the GPU (see below).
 */
#ifndef ATTN_H
#define ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = -1,     /* a null pointer, a non-positive size, misalignment, bad scale */
    ATTN_ERR_UNSUPPORTED = -2, /* a head dim or dtype the library has no kernel for */
    ATTN_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed (launch, tensor map) */
    ATTN_ERR_TIMEOUT = -4,     /* a kernel barrier wait ran out of time; outputs undefined */
    ATTN_ERR_DEVICE = -5       /* no usable sm_103 device */
} attn_status_t;

/*
 * attn_fwd -- the fused forward pass described above, launched on `stream`.
 * Returns ATTN_OK once the kernel is enqueued.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             const uint32_t *mask_bits, int B, int Hq, int Hkv, int S, int d, int causal,
             float scale, int dtype, void *stream);

/*
 * attn_fwd_ex -- the same computation with the generalisations a prefill against a
 * key/value cache and local attention need (the pages themselves stop at Sq = Sk and the
 * masks above; these follow the same tile, bit-word and skip path):
 *   - Sq query rows against Sk >= Sq keys, aligned at the bottom right: query i sits at
 *     key position pos(i) = i + Sk - Sq.  q, o: [B][Hq][Sq][d]; k, v: [B][Hkv][Sk][d];
 *     lse: [B][Hq][Sq].
 *   - a band of kept keys: pos(i) - window_left <= j <= pos(i) + window_right
 *     (-1 = unbounded on that side); causal = 1 keeps j <= pos(i) (window_right is then
 *     treated as 0).
 *   - custom masks of [B][Sq][ceil(Sk/32)] words (mask_per_head = 0) or
 *     [B][Hq][Sq][ceil(Sk/32)] (mask_per_head = 1), ANDed with the band.
 *   - visited: as for attn_fwd_visited (nqt = ceil(Sq/bm), nkt = ceil(Sk/bn)), or NULL.
 *   - variable-length batches: seqlens_q / seqlens_k, int32 [B] in device memory (4-byte
 *     aligned) or NULL (= Sq / Sk for every entry), give batch entry b its own lengths
 *     sq_b <= Sq and sk_b <= Sk inside the padded buffers above (values outside [0, Sq] /
 *     [0, Sk] are clamped).  Entry b's query i sits at key position i + sk_b - sq_b, only
 *     keys j < sk_b exist, and rows i >= sq_b of o and lse are not written.  Key rows at or
 *     past sk_b get weight exactly 0, so v must hold finite values there (0 * inf is NaN);
 *     k there may hold anything.  The custom-mask layout keeps the padded shape.
 *   - packed variable-length batches: cu_seqlens_q / cu_seqlens_k, int32 [B+1] in device
 *     memory (4-byte aligned, non-decreasing, cu[0] = 0), or NULL.  When given, entry b is
 *     query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] ..
 *     cu_seqlens_k[b+1]-1 of head-major packed buffers: q, o: [Hq][Sq][d], k, v:
 *     [Hkv][Sk][d], lse: [Hq][Sq], with Sq / Sk the total row counts; max_seqlen_q /
 *     max_seqlen_k (>= 1) bound every entry's lengths (longer entries are cut to them).
 *     Alignment, causal and window rules are per entry as above; visited is
 *     [B][Hq][ceil(max_seqlen_q/bm)][ceil(max_seqlen_k/bn)].  Custom masks are not supported
 *     with packed layouts (ATTN_ERR_UNSUPPORTED); seqlens_q / seqlens_k must then be NULL.
 * With Sq = Sk = S, windows -1, mask_per_head = 0 and no lengths it is attn_fwd.  Custom masks take
 * stream-ordered scratch of the custom-mask scratch size above.  Errors as for attn_fwd;
 * Sk < Sq is ATTN_ERR_INVALID for padded layouts.
 */
typedef struct {
    const void *q, *k, *v;
    void *o;
    float *lse;
    const uint32_t *mask_bits;
    int mask_per_head;
    int B, Hq, Hkv, Sq, Sk, d;
    int causal, window_left, window_right;
    float scale;
    int dtype;
    void *stream;
    uint8_t *visited;
    const int *seqlens_q, *seqlens_k;
    const int *cu_seqlens_q, *cu_seqlens_k;
    int max_seqlen_q, max_seqlen_k;
} attn_fwd_params_t;

int attn_fwd_ex(const attn_fwd_params_t *params);

/*
 * attn_fwd_visited -- attn_fwd that also records which (query tile, key tile)
 * blocks it computed: visited[((b*Hq + hq)*nqt + qt)*nkt + kt] = 1, uint8,
 * device memory, nqt = ceil(S/bm), nkt = ceil(S/bn) with (bm, bn) from
 * attn_tile_shape.  The caller zeroes `visited`.  Blocks that hold no kept
 * entry -- every mask word over the block is zero, or the block lies above the
 * causal diagonal -- are skipped, following the tile-skip ballot of the page
 * "Opus 4.6 + AutoResearch驱动25轮迭代..." (first code excerpt).  With a custom mask
 * qt numbers the compacted query tiles instead: tile qt holds the 16-row blocks
 * 8*qt .. 8*qt+7 of the ascending list of blocks that keep anything (of batch
 * entry b, or of head (b, hq) for per-head masks).  O and LSE are identical to
 * attn_fwd's.
 */
int attn_fwd_visited(const void *q, const void *k, const void *v, void *o, float *lse,
                     const uint32_t *mask_bits, int B, int Hq, int Hkv, int S, int d,
                     int causal, float scale, int dtype, void *stream, uint8_t *visited);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that must not allocate device memory:
 * code running where cudaMalloc / cudaMallocAsync are unavailable or forbidden,
 * e.g. inside a custom allocator or memory-pool hook (re-entering the allocator
 * would deadlock or recurse), in real-time paths that may not wait on the
 * allocator, or in hosts that hand out a fixed memory budget up front.  It takes
 * the same arguments and computes the same result as attn_fwd.  Without a custom
 * mask the two are the same call.  With one, the mask pre-pass output goes into a
 * fixed device array of ATTN_NOALLOC_SCRATCH_BYTES that this library reserves on
 * every GPU that loads it, held until the process exits, instead of into
 * stream-ordered scratch; calls whose custom-mask scratch size (see the
 * conventions above) exceeds it return ATTN_ERR_INVALID before any launch.
 * Every call looks the array's device address up with the caller's device
 * current (a cheap host call, so a reset or replaced context never sees a stale
 * address); the first call on a device also loads the library's device code
 * there, so make it before any stream capture.  Every call shares the one array
 * and it keeps the last call's contents (each call rewrites every byte it then
 * reads, so nothing needs clearing); calls whose work overlaps on the GPU -- on
 * different streams, say -- race on it, so order them.  It makes no host-side
 * allocation either: on a stream that attn_fwd has not used, its timeout status
 * goes to the status word shared by such streams, which attn_check reports for
 * any of them.  The pages this library follows have no counterpart of this
 * entry point.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (4u << 20)
int attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                     const uint32_t *mask_bits, int B, int Hq, int Hkv, int S, int d, int causal,
                     float scale, int dtype, void *stream);

/*
 * attn_check -- read (and clear) the status word of `stream` on the current
 * device, in stream order after the work enqueued on it so far, and synchronise
 * the stream: ATTN_OK, ATTN_ERR_TIMEOUT if a launch on this stream gave up on a
 * barrier wait, or ATTN_ERR_CUDA if the stream itself reports an error.  Launches
 * on other streams do not affect it (streams share a word only past the first
 * 1023 distinct streams of a device, and for attn_fwd_noalloc calls on streams
 * attn_fwd has not used).
 */
int attn_check(void *stream);

/*
 * attn_release_workspace -- free (in stream order, cudaFreeAsync on `stream`) the
 * custom-mask workspace the library holds for `stream` on the current device, if
 * any.  Call it before destroying a stream that ran custom masks; a later call on
 * the stream simply allocates a new one.  ATTN_OK, or ATTN_ERR_CUDA.
 */
int attn_release_workspace(void *stream);

/*
 * attn_debug_counters -- host-side counters since the library was loaded, for
 * tests and tuning: out[0] = workspace allocations, out[1] = tensor maps encoded,
 * out[2] = tensor maps served from the cache; entries past 2 are set to 0.
 * n = the number of entries of `out` (>= 1).
 */
int attn_debug_counters(unsigned long long *out, int n);

/* attn_strerror -- a static, human-readable string for a status code. */
const char *attn_strerror(int status);

/*
 * attn_tile_shape -- rows per query tile (*bm) and key columns per tile (*bn)
 * the kernel uses for head dim d, i.e. the granularity of tile skipping.
 * Returns ATTN_ERR_UNSUPPORTED for a head dim without a kernel.
 */
int attn_tile_shape(int d, int *bm, int *bn);

/*
 * attn_set_wait_timeout_ns -- the longest a kernel thread waits on one
 * barrier before it abandons the launch and records ATTN_ERR_TIMEOUT
 * (default 2e9 ns).  Applies to launches made after the call.  0 restores the
 * default.
 */
int attn_set_wait_timeout_ns(unsigned long long ns);

/*
 * attn_debug_inject -- test hook.  With flag 1 the next launch's load warp
 * never signals its first query tile, so the consumers' waits run out and the
 * launch ends with ATTN_ERR_TIMEOUT (no fault, no hang: every wait is bounded).
 * The flag clears itself after one launch.  0 disarms it.
 */
int attn_debug_inject(int flag);

/* attn_version -- library version, major*10000 + minor*100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
