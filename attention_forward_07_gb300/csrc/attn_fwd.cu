// attn_fwd.cu -- fused attention forward for GB300 (sm_103a) and the C-ABI of libattn.so.
//
// O = softmax(scale * Q K^T + mask) V and LSE, tile by tile with a running max and
// running sum (the FlashAttention scheme of the page "NVIDIA让AI狂肝7天自己写算子",
// FlashAttention-lineage section), so the S x S scores never leave the SM.
//
// One persistent CTA per SM, 384 threads, warp-specialised:
//   warp 0       load warp: TMA loads of the two 128-row Q tiles of a work unit and of
//                the K / V tiles into a ring of 128-byte-swizzled shared-memory slots;
//                for custom masks it also stages the tile's kept-bit words in shared
//                memory and decides, with a warp ballot over the block flags, which
//                (Q tile, K tile) blocks hold a kept entry (the tile-skip ballot of the
//                page "Opus 4.6 + AutoResearch驱动25轮迭代...", first excerpt).  Empty
//                blocks are never loaded or computed.
//   warp 1       MMA warp: one thread issues tcgen05.mma.  S_t = Q_t K^T (both operands in
//                shared memory, fp32 accumulator in TMEM) and O_t += P_t V (P_t read from
//                TMEM, V from shared memory), interleaved so the QK^T of the next key tile
//                of a Q tile is queued right behind that tile's P.V.
//   warps 4-7,   softmax warpgroups, one per Q tile, one thread per query row (= TMEM
//   8-11         lane): load the 128 scores of the row, scale, mask (causal bound or
//                staged bit words, as in the page's in-register mask excerpt), row max,
//                exp2, row sum, write P back into TMEM as fp16/bf16, rescale the O row
//                when the running max grew (the correction step), and at the end of the
//                unit normalise O, store it and the LSE.
// Work unit = (batch, query head, 256-row block).  Units without a custom mask and
// variable-length batches come from a work queue per stream (an atomic counter the last CTA
// resets): causal ones longest first (block level descending), variable-length ones in the
// longest-first order a one-CTA counting sort writes.  Custom-mask units and windows narrower
// than 1024 keys are dealt in a fixed snake order, the heaviest blocks first.
// d = 64 keeps three S slots in TMEM shared by the two Q tiles, so a Q tile's next Q.K^T runs
// while its softmax works on the current one.
// Custom masks go through two small kernels first: the pre-pass ANDs the caller's words
// with the causal / window / length bounds into whole-tile words (or, when no bound applies
// and the words already fill whole tiles, leaves the kernel to read the caller's) and flags
// each (16-row block, key tile) pair that keeps anything; the compaction lists the 16-row
// blocks that keep anything.  A unit then computes the next sixteen listed blocks as its two
// Q tiles (gathered block by block, or loaded whole when they are its own rows) and writes
// O = 0, LSE = -inf for the rows of its own blocks that keep nothing.  Both kernels let the next
// grid start early (programmatic dependent launch) and the attention kernel waits for
// their output with griddepcontrol.wait.
// Every barrier wait is bounded: a wait that runs out sets a shared abort flag and the
// launch's per-stream status word, every role drains what it has in flight and the CTA
// returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <memory>
#include <mutex>
#include <unordered_map>

#include "attn.h"
#include "ptx.cuh"

namespace attn {

constexpr int BM = 128;        // query rows per Q tile = TMEM lanes
constexpr int QT = 2;          // Q tiles per work unit
constexpr int UNIT_ROWS = BM * QT;
constexpr int BN = 128;        // keys per K/V tile
constexpr int NTHREADS = 384;  // 12 warps
constexpr int REGS_LAUNCH = 168;
constexpr int NINFO = 4;       // depth of the tile-descriptor ring
constexpr int TMEM_COLS = 512;
constexpr int FLAG_END = 4;    // info entry marking the end of a work unit
constexpr int FLAG_EXIT = 8;   // info entry telling the consumers that no unit is left
constexpr float LN2 = 0.69314718055994530942f;

// NONE: every key; CAUSAL: keys up to the aligned position; BAND: keys in
// [key_lo(i), key_hi(i)) per query row (sliding windows); CUSTOM: kept-bit words from the
// mask pre-pass (which folds any band in).  The first two keep their bounds cheap.
enum MaskMode { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_CUSTOM = 2, MASK_BAND = 3 };

template <int D, int MODE>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int HALVES = D / 64;                  // 128-byte swizzle spans per row
  static constexpr int Q_TILE_BYTES = BM * D * 2;
  static constexpr int KV_TILE_BYTES = BN * D * 2;
  // d = 64 (short sequences, many units per CTA) double-buffers the Q tiles so the next
  // unit's Q load overlaps the current unit; d = 128 spends that room on K/V slots.
  static constexpr int QBUF = (D == 64) ? 2 : 1;
  // With two Q buffers a unit's buffer is not refilled before the unit after next, so its
  // epilogue can stage O there and write it out coalesced (8 softmax warps x 32 rows x d
  // fp16/bf16 = exactly one buffer); the buffer is released when those warps are done.
  static constexpr bool STAGE_O = (QBUF == 2);
  static constexpr int QEMPTY_COUNT = 1 + (STAGE_O ? QT * 4 : 0);  // MMA commit + softmax warps
  // TMEM.  d = 128: S_t (fp32, 128 columns) at t * 128, P_t (fp16/bf16 pairs) over its first 64
  // columns, O_t at 256 + t * 128.  d = 64: a ring of three S slots at 0, 128, 256 shared by the
  // two Q tiles (the n-th Q.K^T of the CTA goes to slot n % 3, its P over the slot's first 64
  // columns), O_t at 384 + t * 64: a Q tile's next Q.K^T runs while its softmax works on the
  // current one.
  static constexpr bool RING = (D == 64);
  static constexpr int S_SLOTS = RING ? 3 : QT;
  static constexpr int O_COL = RING ? 384 : 256;
  static constexpr int O_STRIDE = RING ? 64 : 128;
  static_assert(S_SLOTS * 128 + QT * O_STRIDE <= TMEM_COLS, "TMEM columns");
  // Registers per thread after setmaxnreg: the load / MMA warpgroup and the two softmax
  // warpgroups share the launch's 384 x 168 (the ring bookkeeping of d = 64 costs the MMA
  // warp a few; its softmax, with a 64-column O, needs fewer).
  static constexpr int REGS_LOADMMA = (D == 64) ? 96 : 88;
  static constexpr int REGS_SOFTMAX = (D == 64) ? 200 : 208;
  static_assert(128 * REGS_LOADMMA + 256 * REGS_SOFTMAX <= NTHREADS * REGS_LAUNCH, "register split");
  // With one Q buffer (d = 128) the epilogue stages O through a 32 KiB area of its own,
  // 4 KiB per softmax warp, one 64-column half at a time (custom masks need that room for
  // their mask words and write O directly).
  static constexpr bool STAGE_SEP = (D == 128 && MODE != MASK_CUSTOM);
  static constexpr int STAGE_BYTES = STAGE_SEP ? QT * 4 * 32 * 128 : 0;
  // Separate K and V rings: K(j) is read by the two QK^T of tile j, V(j) by the two P.V
  // one tile later, so each ring is released right after its own last reader.
  static constexpr int KSLOT = (D == 128) ? 2 : 4;
  static constexpr int VSLOT = (D == 128) ? 2 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int Q_BUF_BYTES = QT * Q_TILE_BYTES;
  static constexpr int OFF_K = OFF_Q + QBUF * Q_BUF_BYTES;
  static constexpr int OFF_V = OFF_K + KSLOT * KV_TILE_BYTES;
  static constexpr int OFF_STAGE = OFF_V + VSLOT * KV_TILE_BYTES;
  static constexpr int OFF_WORDS = OFF_STAGE + STAGE_BYTES;
  static constexpr int WORDS_PER_ENTRY = UNIT_ROWS * (BN / 32);
  static constexpr int OFF_HDR = OFF_WORDS + (MODE == MASK_CUSTOM ? NINFO * WORDS_PER_ENTRY * 4 : 0);
  static constexpr int OFF_BAR = OFF_HDR + NINFO * 32;
  // barrier indices
  static constexpr int B_QFULL = 0, B_QEMPTY = QBUF, B_KFULL = 2 * QBUF,
                       B_KEMPTY = B_KFULL + KSLOT, B_VFULL = B_KEMPTY + KSLOT,
                       B_VEMPTY = B_VFULL + VSLOT, B_IFULL = B_VEMPTY + VSLOT,
                       B_IEMPTY = B_IFULL + NINFO,
                       B_STILE = B_IEMPTY + NINFO, B_PREADY = B_STILE + S_SLOTS,
                       B_ODONE = B_PREADY + QT, B_OPV = B_ODONE + QT, B_DRAIN = B_OPV + QT,
                       NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
  static_assert(SMEM_ALLOC <= 232448, "shared memory");
  // Over half of the SM's shared memory: one CTA per SM, so TMEM (512 columns) never
  // has to be shared between resident CTAs.
  static_assert(SMEM_ALLOC > 116 * 1024, "one CTA per SM");
};

struct InfoHdr {
  int j;      // key tile index
  int flags;  // bit t: Q tile t computes this key tile; FLAG_END: end of unit
  int sq, sk;  // the unit's query and key lengths (per batch entry with seqlens arrays)
  int qoff;    // packed layouts: the entry's first row in q / o / lse
  int bh, qb;  // the work unit this entry belongs to: b * Hq + hq, 256-row block
  int pad;
};
static_assert(sizeof(InfoHdr) == 32, "descriptor slot size");

struct Params {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps {d, S, B*H}, box {64, 128, 1}, 128B swizzle
  CUtensorMap tm_m;              // kept-bit words {W4, S, nmb}, box {4, 16, 1} (custom masks)
  CUtensorMap tm_q16;            // Q with 16-row boxes: gathers of compacted row blocks
  CUtensorMap tm_m256;           // kept-bit words, box {4, 256, 1}: a unit whose slots are in place
  void* o;
  float* lse;
  // Custom masks (written by the mask kernels): the query rows of a mask row block mb with
  // any kept entry, in 16-row blocks listed in ascending order and packed into 128-row
  // compacted tiles; a work unit (b, hq, qb) computes compacted tiles 2 qb and 2 qb + 1 and
  // owns the 16-row blocks of original rows [256 qb, 256 qb + 256) with nothing kept.
  const uint8_t* tflags;  // [nmb][nqt][nkt] 1 = compacted tile holds a kept entry in key tile
  const int* rowmap;      // [nmb][nqb * 16] original 16-row block of each compacted slot, -1 past the list
  const uint8_t* live;    // [nmb][nr16] 1 = the 16-row block holds a kept entry
  int nr16;               // ceil(Sq / 16)
  uint8_t* visited;
  int B, Hq, Hkv, Sq, Sk, g, nqb, nkt, nqt, W, num_units;
  // Query row i of a batch entry with sq queries and sk keys sits at key position
  // i + off, off = sk - sq (bottom-right alignment); the band keeps keys with
  // pos - wl <= key <= pos + er (wl / er = -1: unbounded).
  int wl, er;
  int mask_heads;  // custom-mask rows per batch entry: Hq (per-head masks) or 1
  const int* lens_q;  // per batch entry query / key lengths inside the padded buffers,
  const int* lens_k;  // clamped to [0, Sq] / [0, Sk]; NULL = Sq / Sk
  // Packed layouts (cu_q != NULL): entry b holds rows cu_q[b] .. cu_q[b+1]-1 of q / o / lse
  // ([Hq][q_rows][d]) and keys cu_k[b] .. cu_k[b+1]-1 of k / v ([Hkv][k_rows][d]); Sq / Sk
  // are then the longest entry's lengths.
  const int* cu_q;
  const int* cu_k;
  int q_rows, k_rows;
  int causal;      // the band only bounds keys on the right: longest units first
  int inject;
  int status_slot;  // index into g_attn_status of the stream this launch runs on
  int dynamic;      // 1: units are taken from the slot's work queue (g_sched), else a fixed walk
  // Variable-length batches with the work queue: the (batch entry, 256-row block) pairs in the
  // order they are handed out, most key tiles first (written by unit_order_kernel); the query
  // heads of a pair follow one another.  NULL: the order decode_unit computes.
  const int* order;
  // 1 when Sq <= 128 and the GQA group size is even (no custom mask): a unit is a pair of query
  // heads (hq, hq + 1) of one K/V head, Q tile t holding rows 0..127 of head hq + t, so both
  // softmax warpgroups work on one stream of K/V tiles; 0: Q tile t holds rows 128 t.. of hq.
  int pair;
  float scale_log2;
  uint32_t timeout_us;  // longest barrier wait (microseconds; 32 bits keep it in one register)
};

}  // namespace attn

// Device status words, one per stream slot (the host gives every (device, stream) pair a
// slot; streams beyond the table share slot 0): bit 0 = a barrier wait ran out of time.
constexpr int STATUS_SLOTS = 1024;
__device__ unsigned int g_attn_status[STATUS_SLOTS];
// Work queue per stream slot: [2 s] = next unit to hand out, [2 s + 1] = CTAs that have
// finished.  Launches on one stream run one after the other, so a slot serves one launch at
// a time; its last CTA resets both words for the next launch.
__device__ unsigned int g_sched[2 * STATUS_SLOTS];

namespace attn {

// Slow path of a bounded barrier wait (inlined: a shared non-inlined callee cannot serve
// warps running under different setmaxnreg budgets).  Gives up when another thread has aborted, when
// the wait has lasted timeout_us, or after an iteration cap, and then aborts the CTA and marks the
// launch's status slot (abort_flag[1], set from the launch parameters at kernel start).
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       uint32_t timeout_us) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > 1000ull * timeout_us) break;
  }
  *abort_flag = 1;
  atomicOr(&g_attn_status[abort_flag[1] & (STATUS_SLOTS - 1)], 1u);
  return false;
}

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      uint32_t timeout_us) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, timeout_us);
}

// Warp-uniform variant: every lane waits, and the warp only proceeds if all lanes did.
__device__ __forceinline__ bool bwait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           uint32_t timeout_us) {
  bool ok = bwait(bar, parity, abort_flag, timeout_us);
  return __all_sync(0xffffffffu, ok);
}

// Wait used only while draining after an abort: ignores the abort flag, short limit.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > 200000000ull) return;
  }
}

// k-th unit of this CTA in the snake order, or -1 when it has none left.
__device__ __forceinline__ int unit_at(int k, int num_units) {
  const int G = gridDim.x;
  const int u = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return u < num_units ? u : -1;
}

// Unit -> (batch, query head, 256-row block).
// Variable-length batches (work queue): the pairs of p.order, longest first, the query heads
// of a pair adjacent.
// Causal: longest first — block index descending, the (batch, head) pairs of a block level
// adjacent.  The work queue hands them out in that order; the fixed walk (custom masks) deals
// them in a snake, so that every CTA's total is close to the mean.
// Custom masks without causal: block level by level from block 0.  Row compaction packs a mask
// row block's kept 16-row blocks into its first units, so this is longest first there too, and
// the snake does not deal the empty units of a sparse mask to every other CTA.
// Otherwise: consecutive units walk the blocks and the query heads of one K/V head, so the
// CTAs running at one time share K/V through L2.
__device__ __forceinline__ void decode_unit(int u, const Params& p, bool causal, bool pair, bool custom, int& b,
                                            int& hq, int& qb) {
  if (pair) {
    // (entry, block) pairs in the work order or in index order, then the head pairs of
    // consecutive K/V heads (an even group size keeps a pair inside one group)
    const int hp = p.Hq >> 1, pi = u / hp;
    const int pr = p.order ? __ldg(p.order + pi) : pi;
    b = pr / p.nqb;
    qb = pr - b * p.nqb;
    hq = 2 * (u - pi * hp);
  } else if (p.order) {
    const int pi = u / p.Hq;
    const int pair = __ldg(p.order + pi);
    b = pair / p.nqb;
    qb = pair - b * p.nqb;
    hq = u - pi * p.Hq;
  } else if (causal || custom) {
    const int bh = u % (p.B * p.Hq), level = u / (p.B * p.Hq);
    qb = causal ? p.nqb - 1 - level : level;
    b = bh / p.Hq;
    hq = bh % p.Hq;
  } else {
    const int member = u % p.g;
    const int rest = u / p.g;
    qb = rest % p.nqb;
    const int bk = rest / p.nqb;
    const int hkv = bk % p.Hkv;
    b = bk / p.Hkv;
    hq = hkv * p.g + member;
  }
}

// Query / key lengths of batch entry b and, for packed layouts, its first query and key row
// (off = sk - sq is its bottom-right alignment).
__device__ __forceinline__ void unit_span(const Params& p, int b, int& sq, int& sk, int& qoff, int& koff) {
  if (p.cu_q) {
    qoff = __ldg(p.cu_q + b);
    koff = __ldg(p.cu_k + b);
    sq = min(max(__ldg(p.cu_q + b + 1) - qoff, 0), p.Sq);
    sk = min(max(__ldg(p.cu_k + b + 1) - koff, 0), p.Sk);
  } else {
    qoff = koff = 0;
    sq = p.lens_q ? min(max(__ldg(p.lens_q + b), 0), p.Sq) : p.Sq;
    sk = p.lens_k ? min(max(__ldg(p.lens_k + b), 0), p.Sk) : p.Sk;
  }
}
// Rows of (b, hq) in q / o / lse start here (padded: its own [Sq] block; packed: the entry's
// rows inside head hq's [q_rows] block).
__device__ __forceinline__ size_t q_row_base(const Params& p, int b, int hq, int qoff) {
  return p.cu_q ? (size_t)hq * p.q_rows + qoff : (size_t)(b * p.Hq + hq) * p.Sq;
}
__device__ __forceinline__ void unit_lengths(const Params& p, int b, int& sq, int& sk) {
  sq = p.lens_q ? min(max(__ldg(p.lens_q + b), 0), p.Sq) : p.Sq;
  sk = p.lens_k ? min(max(__ldg(p.lens_k + b), 0), p.Sk) : p.Sk;
}

// Kept keys of query row i under the band: [key_lo, key_hi) (empty when hi <= lo).
__device__ __forceinline__ int key_lo(const Params& p, int i, int off) {
  return p.wl < 0 ? 0 : max(0, i + off - p.wl);
}
__device__ __forceinline__ int key_hi(const Params& p, int i, int off, int sk) {
  return p.er < 0 ? sk : min(sk, i + off + p.er + 1);
}

}  // namespace attn

namespace attn {

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// ------------------------------------------------------------------ load warp (warp 0)
template <int D, bool BF16, int MODE>
__device__ __forceinline__ void load_role(const Params& p, uint32_t base, uint8_t* gbase,
                                          volatile int* abort_flag, int lane) {
  using L = Layout<D, MODE>;
  const bool causal = (MODE == MASK_CAUSAL) || (MODE != MASK_NONE && p.causal != 0);
  const bool pair = MODE != MASK_CUSTOM && p.pair;  // head pairs never come with a custom mask
  const uint32_t to = p.timeout_us;
  const uint32_t bars = base + L::OFF_BAR;
  volatile InfoHdr* hdr = reinterpret_cast<volatile InfoHdr*>(gbase + L::OFF_HDR);

  uint32_t q_empty_par = (1u << L::QBUF) - 1u;  // per Q buffer; "empty" waits start at parity 1
  uint32_t q_pend = 0, q_pend_par = 0;           // Q buffers with a load issued, its full parity
  // ring position and "empty" parity of the K and V rings; loads issued but possibly not
  // landed (bit per slot) and the full-barrier parity each of those loads completes
  int kslot = 0, vslot = 0;
  uint32_t kpar = 1, vpar = 1;
  uint32_t kpend = 0, kpend_par = 0, vpend = 0, vpend_par = 0;
  int ie = 0;
  uint32_t ie_par = 1;
  uint32_t ipend = 0, ipend_par = 0;  // descriptor slots with a mask-word load issued
  bool inject = p.inject != 0;

  // The work queue: lane 0 fetches the index of the unit after the current one as the current
  // one starts, so the atomic's round trip to L2 overlaps the current unit's loads.
  unsigned int q_next = 0;
  if (p.dynamic && lane == 0) q_next = atomicAdd(&g_sched[2 * p.status_slot], 1u);
  for (int k = 0;; ++k) {
    int u;
    if (p.dynamic) {
      const unsigned int x = __shfl_sync(0xffffffffu, q_next, 0);
      u = x < (unsigned int)p.num_units ? (int)x : -1;
      if (u >= 0 && lane == 0) q_next = atomicAdd(&g_sched[2 * p.status_slot], 1u);
    } else {
      u = unit_at(k, p.num_units);
    }
    if (u < 0) {
      // no unit left: an exit descriptor releases the MMA warp and the softmax warpgroups
      if (!bwait_warp(bars + 8u * (L::B_IEMPTY + ie), ie_par, abort_flag, to)) goto drain;
      if (lane == 0) {
        hdr[ie].j = -1;
        hdr[ie].flags = FLAG_EXIT;
        mbar_arrive(bars + 8u * (L::B_IFULL + ie));
      }
      __syncwarp();
      if (++ie == NINFO) { ie = 0; ie_par ^= 1u; }
      break;
    }
    int b, hq, qb;
    decode_unit(u, p, causal, pair, MODE == MASK_CUSTOM, b, hq, qb);
    const int hkv = hq / p.g;
    const int row0 = qb * UNIT_ROWS;
    const int mb = p.mask_heads > 1 ? b * p.Hq + hq : b;  // custom-mask row block
    // Custom masks: lane s < 16 holds the original 16-row block of compacted slot s of the
    // unit (-1: none), and the unit has nothing to compute when its first slot is empty.
    int slot_blk = -1;
    bool unit_empty = false, in_place = true;
    if constexpr (MODE == MASK_CUSTOM) {
      if (lane < 2 * QT * 4) slot_blk = __ldg(p.rowmap + ((size_t)mb * p.nqb + qb) * 16 + lane);
      unit_empty = __shfl_sync(0xffffffffu, slot_blk, 0) < 0;
      // slots that are the unit's own rows (no empty block among them): plain tile loads
      const int own = qb * 16 + lane;
      in_place = __all_sync(0xffffffffu, lane >= 2 * QT * 4 || slot_blk == (own < p.nr16 ? own : -1));
    }

    int sq, sk, qoff, koff;
    unit_span(p, b, sq, sk, qoff, koff);
    const int qz = p.cu_q ? hq : b * p.Hq + hq, kz = p.cu_q ? hkv : b * p.Hkv + hkv;  // TMA z

    // Both Q tiles of the unit (rows past S are zero-filled by the TMA unit).  Custom masks
    // gather them block by block from the compacted list (a missing block reads as zeros).
    const int qbuf = k % L::QBUF;
    if (!bwait_warp(bars + 8u * (L::B_QEMPTY + qbuf), (q_empty_par >> qbuf) & 1u, abort_flag, to))
      goto drain;
    q_empty_par ^= 1u << qbuf;
    if (!inject) {
      const uint32_t fb = bars + 8u * (L::B_QFULL + qbuf);
      if (MODE == MASK_CUSTOM && !in_place) {
        if (lane == 0) mbar_expect_tx(fb, unit_empty ? 0u : (uint32_t)L::Q_BUF_BYTES);
        __syncwarp();
        if (!unit_empty && lane < 2 * QT * 4) {
          const int t = lane >> 3, blk = lane & 7;
          const int y = slot_blk >= 0 ? slot_blk * 16 : p.Sq;  // past Sq: zero fill
#pragma unroll
          for (int h = 0; h < L::HALVES; ++h)
            tma_load_3d(base + L::OFF_Q + qbuf * L::Q_BUF_BYTES + t * L::Q_TILE_BYTES + h * BM * 128 + blk * 16 * 128,
                        &p.tm_q16, fb, h * 64, y, b * p.Hq + hq);
        }
      } else if (lane == 0) {
        mbar_expect_tx(fb, L::Q_BUF_BYTES);
#pragma unroll
        for (int t = 0; t < QT; ++t)
#pragma unroll
          for (int h = 0; h < L::HALVES; ++h)
            tma_load_3d(base + L::OFF_Q + qbuf * L::Q_BUF_BYTES + t * L::Q_TILE_BYTES + h * BM * 128,
                        &p.tm_q, fb, h * 64, qoff + row0 + (pair ? 0 : t * BM), qz + (pair ? t : 0));
      }
      // this fill completes the phase the consumer waits for with parity (empty parity ^ 1)
      q_pend |= 1u << qbuf;
      q_pend_par = (q_pend_par & ~(1u << qbuf)) | ((((q_empty_par >> qbuf) & 1u)) << qbuf);
    }
    inject = false;

    const int off = sk - sq;
    // Key-tile range of each Q tile under the band.  key_lo / key_hi grow by one per row,
    // so the kept keys of rows rf..r1 form the one range [key_lo(rf), key_hi(r1)), rf being
    // the first row whose band is not empty (rows at key position < -er keep nothing).
    int jlo[QT], jhi[QT];
#pragma unroll
    for (int t = 0; t < QT; ++t) {
      const int r0 = row0 + (pair ? 0 : t * BM);
      const int r1 = min(r0 + BM - 1, sq - 1);
      const int rf = p.er >= 0 ? max(r0, -off - p.er) : r0;
      const int klo = key_lo(p, rf, off), khi = key_hi(p, r1, off, sk);
      const bool any = r0 < sq && rf <= r1 && khi > klo;
      jlo[t] = any ? klo / BN : 0;
      jhi[t] = any ? (khi - 1) / BN : -1;  // -1: nothing to compute for this Q tile
      if constexpr (MODE == MASK_CUSTOM) {
        // compacted tiles: every key tile, the flags decide (band and lengths are in them)
        const bool valid = __shfl_sync(0xffffffffu, slot_blk, t * 8) >= 0;
        jlo[t] = 0;
        jhi[t] = valid ? p.nkt - 1 : -1;
      }
    }
    const int jbeg = jhi[0] < 0 ? jlo[1] : (jhi[1] < 0 ? jlo[0] : min(jlo[0], jlo[1]));
    const int jend = max(jhi[0], jhi[1]) + 1;
    uint32_t f0 = 0, f1 = 0;  // bit (j % 32): Q tile 0 / 1 has a kept entry in key tile j
    // Causal: odd block levels walk their key tiles from the diagonal down.  Longest first, a
    // head's next-lower level starts about when its current one ends, so it begins on the K/V
    // tiles that level read last (still in L2) rather than on its oldest ones.  The online
    // softmax does not depend on the order of the key tiles.
    const bool down = MODE == MASK_CAUSAL && (qb & 1);
    for (int jj = jbeg; jj < jend; ++jj) {
      const int j = down ? jend - 1 - (jj - jbeg) : jj;
      bool a0 = j >= jlo[0] && j <= jhi[0];
      bool a1 = j >= jlo[1] && j <= jhi[1];
      if constexpr (MODE == MASK_CUSTOM) {
        // Emptiness bits of the two compacted Q tiles for 32 key tiles at a time, from the
        // map the mask kernels wrote (exact: custom bits AND band AND lengths).
        if (j == jbeg || (j & 31) == 0) {
          const int jj = (j & ~31) + lane;
          const size_t fb = ((size_t)mb * p.nqt + qb * QT) * p.nkt;
          uint32_t x0 = 0, x1 = 0;
          if (jj < p.nkt) {
            x0 = p.tflags[fb + jj];
            if (qb * QT + 1 < p.nqt) x1 = p.tflags[fb + p.nkt + jj];
          }
          f0 = __ballot_sync(0xffffffffu, x0 != 0u);
          f1 = __ballot_sync(0xffffffffu, x1 != 0u);
        }
        a0 = a0 && ((f0 >> (j & 31)) & 1u);
        a1 = a1 && ((f1 >> (j & 31)) & 1u);
      }
      if (!a0 && !a1) continue;  // empty block pair: nothing loaded, nothing computed

      if (!bwait_warp(bars + 8u * (L::B_IEMPTY + ie), ie_par, abort_flag, to)) goto drain;
      if (lane == 0) {
        hdr[ie].j = j;
        hdr[ie].flags = (a0 ? 1 : 0) | (a1 ? 2 : 0);
        hdr[ie].sq = sq;
        hdr[ie].sk = sk;
        hdr[ie].qoff = qoff;
        hdr[ie].bh = b * p.Hq + hq;
        hdr[ie].qb = qb;
        const uint32_t fb = bars + 8u * (L::B_IFULL + ie);
        if constexpr (MODE == MASK_CUSTOM) {
          mbar_expect_tx(fb, L::WORDS_PER_ENTRY * 4);
        } else {
          mbar_arrive(fb);
        }
      }
      if constexpr (MODE == MASK_CUSTOM) {
        // the kept-bit words of the unit's 16 compacted slots (16 rows x 4 words each) land
        // in the descriptor slot in compacted row order; a missing block reads as zeros
        __syncwarp();
        const uint32_t wdst = base + L::OFF_WORDS + ie * L::WORDS_PER_ENTRY * 4;
        if (in_place) {
          if (lane == 0) tma_load_3d(wdst, &p.tm_m256, bars + 8u * (L::B_IFULL + ie), j * (BN / 32), row0, mb);
        } else if (lane < 2 * QT * 4) {
          tma_load_3d(wdst + lane * 16 * (BN / 32) * 4, &p.tm_m, bars + 8u * (L::B_IFULL + ie), j * (BN / 32),
                      slot_blk >= 0 ? slot_blk * 16 : p.Sq, mb);
        }
      }
      if constexpr (MODE == MASK_CUSTOM) {
        ipend |= 1u << ie;
        ipend_par = (ipend_par & ~(1u << ie)) | ((ie_par ^ 1u) << ie);
      }
      __syncwarp();
      if (++ie == NINFO) { ie = 0; ie_par ^= 1u; }

      // K tile j
      if (!bwait_warp(bars + 8u * (L::B_KEMPTY + kslot), kpar, abort_flag, to)) goto drain;
      if (lane == 0) {
        const uint32_t fb = bars + 8u * (L::B_KFULL + kslot);
        mbar_expect_tx(fb, L::KV_TILE_BYTES);
#pragma unroll
        for (int h = 0; h < L::HALVES; ++h)
          tma_load_3d(base + L::OFF_K + kslot * L::KV_TILE_BYTES + h * BN * 128, &p.tm_k, fb,
                      h * 64, koff + j * BN, kz);
      }
      kpend |= 1u << kslot;
      kpend_par = (kpend_par & ~(1u << kslot)) | ((kpar ^ 1u) << kslot);
      if (++kslot == L::KSLOT) { kslot = 0; kpar ^= 1u; }
      // V tile j
      if (!bwait_warp(bars + 8u * (L::B_VEMPTY + vslot), vpar, abort_flag, to)) goto drain;
      if (lane == 0) {
        const uint32_t fb = bars + 8u * (L::B_VFULL + vslot);
        mbar_expect_tx(fb, L::KV_TILE_BYTES);
#pragma unroll
        for (int h = 0; h < L::HALVES; ++h)
          tma_load_3d(base + L::OFF_V + vslot * L::KV_TILE_BYTES + h * BN * 128, &p.tm_v, fb,
                      h * 64, koff + j * BN, kz);
      }
      vpend |= 1u << vslot;
      vpend_par = (vpend_par & ~(1u << vslot)) | ((vpar ^ 1u) << vslot);
      if (++vslot == L::VSLOT) { vslot = 0; vpar ^= 1u; }
    }
    // End-of-unit marker.
    if (!bwait_warp(bars + 8u * (L::B_IEMPTY + ie), ie_par, abort_flag, to)) goto drain;
    if (lane == 0) {
      hdr[ie].j = -1;
      hdr[ie].flags = FLAG_END;
      hdr[ie].sq = sq;
      hdr[ie].sk = sk;
      hdr[ie].qoff = qoff;
      hdr[ie].bh = b * p.Hq + hq;
      hdr[ie].qb = qb;
      mbar_arrive(bars + 8u * (L::B_IFULL + ie));
    }
    __syncwarp();
    if (++ie == NINFO) { ie = 0; ie_par ^= 1u; }
  }
  return;

drain:
  // Aborted: let the copies this warp started land before the CTA exits.
  if (lane == 0) {
    for (int s = 0; s < L::KSLOT; ++s)
      if ((kpend >> s) & 1u) wait_drain(bars + 8u * (L::B_KFULL + s), (kpend_par >> s) & 1u);
    for (int s = 0; s < L::VSLOT; ++s)
      if ((vpend >> s) & 1u) wait_drain(bars + 8u * (L::B_VFULL + s), (vpend_par >> s) & 1u);
    for (int qb2 = 0; qb2 < L::QBUF; ++qb2)
      if ((q_pend >> qb2) & 1u) wait_drain(bars + 8u * (L::B_QFULL + qb2), (q_pend_par >> qb2) & 1u);
    for (int e = 0; e < NINFO; ++e)
      if ((ipend >> e) & 1u) wait_drain(bars + 8u * (L::B_IFULL + e), (ipend_par >> e) & 1u);
  }
  __syncwarp();
}

}  // namespace attn

namespace attn {

// ------------------------------------------------------------------ MMA issuer (warp 1)
// The whole warp runs this code converged (descriptors in uniform registers); elect.sync
// picks the lane that issues each tcgen05 instruction.  Per tile descriptor e (key tile j)
// and Q tile t:
//   d = 128:  O_t (+)= P_t(prev) . V(prev)   once softmax t has written P for the previous tile,
//             S_t     = Q_t . K(j)^T         then signal softmax t;
//             S_t / P_t share TMEM columns, so S_t is rewritten only after the P.V that reads it.
//   d = 64:   S(n)    = Q_t . K(j)^T         into ring slot n % 3 (the CTA's n-th Q.K^T),
//             O_t (+)= P_t(prev) . V(prev)   from the slot of the previous tile's S,
//             so the next S of a Q tile is computed while its softmax still works on the
//             current one.  At most two slots hold an S or P whose P.V is not yet issued when
//             a Q.K^T is issued, so the third is free; each P.V is followed by a commit on
//             OPV(t), which the softmax waits for before it rescales O_t.
// Each ring slot of K / V is released by a commit right after its last reader.
template <int D, bool BF16, int MODE>
__device__ __forceinline__ void mma_role(const Params& p, uint32_t base, uint8_t* gbase,
                                         volatile int* abort_flag, uint32_t tmem, int lane) {
  using L = Layout<D, MODE>;
  const uint32_t to = p.timeout_us;
  const uint32_t bars = base + L::OFF_BAR;
  volatile InfoHdr* hdr = reinterpret_cast<volatile InfoHdr*>(gbase + L::OFF_HDR);
  constexpr uint32_t ID_QK = idesc_f16acc32(BF16, false, false, BM, BN);
  constexpr uint32_t ID_PV = idesc_f16acc32(BF16, false, true, BM, D);
  const bool pair = MODE != MASK_CUSTOM && p.pair;

  uint32_t q_par = 0, ie_par = 0, kpar = 0, vpar = 0, p_par0 = 0, p_par1 = 0;  // q_par: bit per Q buffer
  int kslot = 0, vslot = 0, ie = 0;
  int nqk = 0;                 // d = 64: ring slot of the next Q.K^T
  int pslot0 = 0, pslot1 = 0;  // d = 64: ring slot holding P_t of the previous key tile

  for (int k = 0;; ++k) {
    // the unit's first descriptor names it (the loop below waits on it again, at once)
    if (!bwait_warp(bars + 8u * (L::B_IFULL + ie), ie_par, abort_flag, to)) goto drain;
    if (hdr[ie].flags & FLAG_EXIT) {
      mbar_arrive_elect(bars + 8u * (L::B_IEMPTY + ie));
      break;
    }
    const int bh = hdr[ie].bh, qb = hdr[ie].qb;
    const int b = bh / p.Hq, hq = bh - b * p.Hq;
    const int qbuf = k % L::QBUF;
    if (!bwait_warp(bars + 8u * (L::B_QFULL + qbuf), (q_par >> qbuf) & 1u, abort_flag, to)) goto drain;
    q_par ^= 1u << qbuf;
    tc_fence_after();

    bool have_prev = false, pv0 = false, pv1 = false;
    int prev_flags = 0, prev_vslot = 0;
    uint32_t prev_vpar = 0;
    while (true) {
      if (!bwait_warp(bars + 8u * (L::B_IFULL + ie), ie_par, abort_flag, to)) goto drain;
      const int j = hdr[ie].j;
      const int flags = hdr[ie].flags;
      const bool end = (flags & FLAG_END) != 0;
      const int cur_kslot = kslot, cur_vslot = vslot;
      const uint32_t cur_kpar = kpar, cur_vpar = vpar;
      if (!end) {
        if (++kslot == L::KSLOT) { kslot = 0; kpar ^= 1u; }
        if (++vslot == L::VSLOT) { vslot = 0; vpar ^= 1u; }
      }
      // End of unit: every Q_t K^T of the unit is in the pipe, so the Q buffer is released
      // (to the next unit's load) before the last P.V, which does not read it.
      if (end) tc_commit_elect(bars + 8u * (L::B_QEMPTY + qbuf));
      if (have_prev) {
        if (!bwait_warp(bars + 8u * (L::B_VFULL + prev_vslot), prev_vpar, abort_flag, to)) goto drain;
        tc_fence_after();
      }
      bool k_ready = false;

#pragma unroll
      for (int t = 0; t < QT; ++t) {
        int& pslot = t ? pslot1 : pslot0;
        int new_slot = t;
#pragma unroll
        for (int step = 0; step < 2; ++step) {
          // d = 64 issues this tile's Q.K^T first, d = 128 its P.V first
          if ((step == 0) == L::RING) {
            if (!end && ((flags >> t) & 1)) {
              if (!k_ready) {
                if (!bwait_warp(bars + 8u * (L::B_KFULL + cur_kslot), cur_kpar, abort_flag, to)) goto drain;
                tc_fence_after();
                k_ready = true;
              }
              if constexpr (L::RING) {
                new_slot = nqk;
                nqk = nqk == L::S_SLOTS - 1 ? 0 : nqk + 1;
              }
              const uint32_t s_col = tmem + new_slot * 128;
              const uint32_t qbase = base + L::OFF_Q + qbuf * L::Q_BUF_BYTES + t * L::Q_TILE_BYTES;
              const uint32_t kbase = base + L::OFF_K + cur_kslot * L::KV_TILE_BYTES;
              // Q and K as K-major operands: 16 elements (32 bytes) per step inside a
              // 128-byte swizzle row, the next 64 elements one half-tile further.
              if constexpr (D == 64) {
                // d = 64 issues twice the instructions per flop: the descriptors are built
                // once and stepped through their start-address field (address >> 4 in the
                // low 14 bits; every offset here keeps it below 2^14)
                const uint64_t qd = sdesc_sw128(qbase, 16, 1024), kd = sdesc_sw128(kbase, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
                  mma_ss_elect(s_col, qd + off, kd + off, ID_QK, kk > 0 ? 1u : 0u);
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                  mma_ss_elect(s_col, sdesc_sw128(qbase + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                               ID_QK, kk > 0 ? 1u : 0u);
                }
              }
              tc_commit_elect(bars + 8u * (L::B_STILE + new_slot));
              if (p.visited && lane == 0)
                p.visited[((size_t)(b * p.Hq + hq + (pair ? t : 0)) * p.nqt + (qb * QT + (pair ? 0 : t))) * p.nkt + j] = 1;
              __syncwarp();
            }
          } else {
            if (have_prev && ((prev_flags >> t) & 1)) {
              uint32_t& pp = t ? p_par1 : p_par0;
              if (!bwait_warp(bars + 8u * (L::B_PREADY + t), pp, abort_flag, to)) goto drain;
              pp ^= 1u;
              tc_fence_after();
              bool& started = t ? pv1 : pv0;
              const uint32_t p_col = tmem + (L::RING ? pslot : t) * 128;
              const uint32_t vbase = base + L::OFF_V + prev_vslot * L::KV_TILE_BYTES;
              // V tile as the MN-major B operand: 16 keys per step (2048 bytes), the two
              // 64-column halves of d are KV_TILE_BYTES/2 apart, 8-key groups 1024 apart.
              if constexpr (D == 64) {
                const uint64_t vd = sdesc_sw128(vbase, BN * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                  mma_ts_elect(tmem + L::O_COL + t * L::O_STRIDE, p_col + kk * 8, vd + (uint64_t)(kk * 16 * 128 >> 4),
                               ID_PV, (started || kk > 0) ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                  mma_ts_elect(tmem + L::O_COL + t * L::O_STRIDE, p_col + kk * 8,
                               sdesc_sw128(vbase + kk * 16 * 128, BN * 128, 1024), ID_PV,
                               (started || kk > 0) ? 1u : 0u);
              }
              started = true;
              if constexpr (L::RING) tc_commit_elect(bars + 8u * (L::B_OPV + t));
            }
            // end of unit: O_t is complete once its last P.V is -- signal it now, so softmax t
            // starts its epilogue without waiting for the other Q tile's P.V
            if (end && (t ? pv1 : pv0)) tc_commit_elect(bars + 8u * (L::B_ODONE + t));
            if (t == QT - 1 && have_prev) tc_commit_elect(bars + 8u * (L::B_VEMPTY + prev_vslot));
          }
        }
        if constexpr (L::RING) {
          if (!end && ((flags >> t) & 1)) pslot = new_slot;
        }
      }
      if (!end) tc_commit_elect(bars + 8u * (L::B_KEMPTY + cur_kslot));
      mbar_arrive_elect(bars + 8u * (L::B_IEMPTY + ie));
      if (++ie == NINFO) { ie = 0; ie_par ^= 1u; }
      if (end) break;
      have_prev = true;
      prev_flags = flags;
      prev_vslot = cur_vslot;
      prev_vpar = cur_vpar;
    }
  }
  return;

drain:
  // Aborted: wait until every MMA this warp issued has finished before TMEM is freed.
  tc_commit_elect(bars + 8u * L::B_DRAIN);
  wait_drain(bars + 8u * L::B_DRAIN, 0);
  __syncwarp();
}

}  // namespace attn

namespace attn {

// ------------------------------------------------------------------ softmax warpgroup t
// Thread r of the warpgroup owns query row qb*256 + t*128 + r, i.e. TMEM lane r.
// Running state in the exp2 domain: m = max of scale*log2(e)*s over the kept keys seen
// so far, l = sum of 2^(scale*log2(e)*s - m).  LSE = ln2 * (m + log2 l).
template <int D, bool BF16, int MODE>
__device__ __forceinline__ void softmax_role(const Params& p, uint32_t base, uint8_t* gbase,
                                             volatile int* abort_flag, uint32_t tmem, int t,
                                             int quarter, int lane) {
  using L = Layout<D, MODE>;
  using OutT = uint16_t;
  const uint32_t to = p.timeout_us;
  const uint32_t bars = base + L::OFF_BAR;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(gbase + L::OFF_WORDS);
  volatile InfoHdr* hdr = reinterpret_cast<volatile InfoHdr*>(gbase + L::OFF_HDR);
  const int r = quarter * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  const uint32_t o_addr = tmem + lane_off + L::O_COL + t * L::O_STRIDE;
  const float c = p.scale_log2;

  uint32_t s_par = 0, o_par = 0, ie_par = 0;
  int ie = 0;
  int nq = 0;  // d = 64: Q.K^T the MMA warp has issued before the current descriptor's
  int np = 0;  // d = 64: P tiles this thread's Q tile has produced (one P.V, one OPV phase each)

  for (int k = 0;; ++k) {
    // the unit's first descriptor names it (the loop below waits on it again, at once)
    if (!bwait_warp(bars + 8u * (L::B_IFULL + ie), ie_par, abort_flag, to)) return;
    if (hdr[ie].flags & FLAG_EXIT) {
      mbar_arrive(bars + 8u * (L::B_IEMPTY + ie));
      break;
    }
    const int bh = hdr[ie].bh, qb = hdr[ie].qb;
    const int b = bh / p.Hq, hq = bh - b * p.Hq;
    const int mb = p.mask_heads > 1 ? b * p.Hq + hq : b;  // custom-mask row block
    // this tile's query head and first row (head pairs: head hq + t, rows from 0)
    const bool pair = MODE != MASK_CUSTOM && p.pair;
    const int hq_t = hq + (pair ? t : 0);
    const int rt = qb * UNIT_ROWS + (pair ? 0 : t * BM);
    // This thread's query row.  Custom masks: the tile holds compacted slots, 16 rows each;
    // blk_a / blk_b are the original blocks of this warp's two slots (-1: no such slot).
    int i = rt + r;
    int blk_a = 0, blk_b = 0;
    bool live_a = true, live_b = true;  // this warp's own two 16-row blocks keep something
    const int hb0 = (qb * UNIT_ROWS + t * BM + quarter * 32) / 16;
    if constexpr (MODE == MASK_CUSTOM) {
      const int* rm = p.rowmap + ((size_t)mb * p.nqb + qb) * 16 + t * 8 + quarter * 2;
      blk_a = __ldg(rm);
      blk_b = __ldg(rm + 1);
      const int blk = lane < 16 ? blk_a : blk_b;
      i = blk >= 0 ? blk * 16 + (lane & 15) : -1;
      if constexpr (D == 64) {
        // read now, used by the epilogue (the loads overlap the unit's first tile; d = 128
        // has no registers to spare and reads them at the epilogue)
        live_a = hb0 >= p.nr16 || __ldg(p.live + (size_t)mb * p.nr16 + hb0) != 0;
        live_b = hb0 + 1 >= p.nr16 || __ldg(p.live + (size_t)mb * p.nr16 + hb0 + 1) != 0;
      }
    }
    float m = -INFINITY, l = 0.f;
    int nact = 0;
    int sq = p.Sq, sk = p.Sk, qoff = 0;  // the unit's lengths and first row, in every descriptor

    while (true) {
      if (!bwait_warp(bars + 8u * (L::B_IFULL + ie), ie_par, abort_flag, to)) return;
      const int j = hdr[ie].j;
      const int flags = hdr[ie].flags;
      sq = hdr[ie].sq;
      sk = hdr[ie].sk;
      qoff = hdr[ie].qoff;
      const bool end = (flags & FLAG_END) != 0;
      const bool act = !end && ((flags >> t) & 1);
      uint4 wv = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (MODE == MASK_CUSTOM) {
        if (act) wv = *reinterpret_cast<const uint4*>(words + ie * L::WORDS_PER_ENTRY + (t * BM + r) * 4);
      }
      mbar_arrive(bars + 8u * (L::B_IEMPTY + ie));
      if (++ie == NINFO) { ie = 0; ie_par ^= 1u; }
      if (end) break;
      // where this tile's S is: its own columns (d = 128), or the ring slot of its Q.K^T
      // (d = 64: the MMA warp issues Q_0 K^T before Q_1 K^T for each descriptor)
      int slot = t;
      uint32_t spar = s_par;
      if constexpr (L::RING) {
        const int before = nq + ((t == 1 && (flags & 1)) ? 1 : 0);
        slot = before % L::S_SLOTS;
        spar = (uint32_t)(before / L::S_SLOTS) & 1u;
        nq += (flags & 1) + ((flags >> 1) & 1);
      }
      if (!act) continue;
      const uint32_t s_addr = tmem + lane_off + slot * 128;

      if (!bwait_warp(bars + 8u * (L::B_STILE + slot), spar, abort_flag, to)) return;
      if constexpr (!L::RING) s_par ^= 1u;
      tc_fence_after();
      // Scores: the first 64 columns are loaded and reduced while the last 64 are in flight.
      uint32_t sr[128];
      uint32_t(&sa)[64] = *reinterpret_cast<uint32_t(*)[64]>(&sr[0]);
      uint32_t(&sb)[64] = *reinterpret_cast<uint32_t(*)[64]>(&sr[64]);
      tmem_ld32x32b_x64_wait(s_addr, sa);
      tmem_ld32x32b_x64(s_addr + 64, sb);

      // Mask: excluded scores become -inf (weight exactly 0).
      // band / key bound: kept columns of this tile are [lo, hi) relative to its first key
      const int off = sk - sq;
      const int hi = (MODE == MASK_NONE ? sk
                      : MODE == MASK_CAUSAL ? min(sk, i + off + 1)
                                            : key_hi(p, i, off, sk)) - j * BN;
      const int lo = (MODE == MASK_BAND) ? key_lo(p, i, off) - j * BN : 0;
      const bool edge = (MODE != MASK_CUSTOM) && __any_sync(0xffffffffu, hi < BN || lo > 0);
      const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
      auto mask_half = [&](uint32_t(&h)[64], int c0) {
        if constexpr (MODE == MASK_CUSTOM) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (!((wa[(c0 + cc) >> 5] >> ((c0 + cc) & 31)) & 1u)) h[cc] = __float_as_uint(-INFINITY);
        } else if (edge) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (c0 + cc >= hi || c0 + cc < lo) h[cc] = __float_as_uint(-INFINITY);
        }
      };
      // Row max of one half: four independent 3-input max chains, chain x over h[16x, 16x+16).
      auto max_half = [&](const uint32_t(&h)[64]) {
        float a4[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          a4[x] = fmaxf(__uint_as_float(h[16 * x]), __uint_as_float(h[16 * x + 1]));
#pragma unroll
          for (int e = 2; e < 16; e += 2)
            a4[x] = fmax3(a4[x], __uint_as_float(h[16 * x + e]), __uint_as_float(h[16 * x + e + 1]));
        }
        return fmax3(a4[0], a4[1], fmaxf(a4[2], a4[3]));
      };
      mask_half(sa, 0);
      const float mx_a = max_half(sa);
      tmem_wait_ld();
      tmem_fence_regs_x64(sb);
      mask_half(sb, 64);
      const float mx = fmaxf(mx_a, max_half(sb));

      // Lazy rescaling: the exponent base m only moves when the row max exceeds it by more
      // than 8 (weights stay <= 2^8); O and l are always scaled with the same base, so the
      // final O / l and LSE = ln2 * (m + log2 l) are exact.
      const float mx_s = mx * c;
      const bool grow = mx_s > m + 8.f;  // also true on the first kept key (m = -inf)
      const float m_new = grow ? mx_s : m;
      const float alpha = grow ? ex2_approx(m - m_new) : 1.f;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;

      // Correction: rescale this row of O (only warps where some row moved its base).
      if (nact > 0 && __any_sync(0xffffffffu, grow)) {
        if constexpr (L::RING) {
          // d = 64: this tile's S was computed before the previous P.V was issued; wait
          // until that P.V (OPV phase np - 1, the latest that can have completed) is done
          if (!bwait_warp(bars + 8u * (L::B_OPV + t), (uint32_t)(np - 1) & 1u, abort_flag, to)) return;
          tc_fence_after();
        }
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int ch = 0; ch < D / 16; ++ch) {
          uint32_t ob[16];
          tmem_ld32x32b_x16_wait(o_addr + ch * 16, ob);
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            float lo, hi;
            f2_unpack(fmul2(f2_pack(__uint_as_float(ob[2 * x]), __uint_as_float(ob[2 * x + 1])), a2), lo, hi);
            ob[2 * x] = __float_as_uint(lo);
            ob[2 * x + 1] = __float_as_uint(hi);
          }
          tmem_st32x32b_x16(o_addr + ch * 16, ob);
        }
      }

      // P = 2^(s*c - m): packed FMA for the arguments, MUFU ex2, four packed partial sums.
      const uint64_t c2 = f2_pack(c, c);
      const uint64_t nm2 = f2_pack(-m_use, -m_use);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      // P_t goes over the first 64 columns of S_t, in four stores so each overlaps the
      // exponentials of the next quarter (and few packed words are live at a time).
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        uint32_t pk[16];
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const int e = hh * 16 + cc;
          float e0, e1;
          f2_unpack(ffma2(f2_pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), c2, nm2), e0, e1);
          const float p0 = ex2_approx(e0);
          const float p1 = ex2_approx(e1);
          acc[cc & 3] = fadd2(acc[cc & 3], f2_pack(p0, p1));
          pk[cc] = pack2<BF16>(p0, p1);
        }
        tmem_st32x32b_x16(s_addr + hh * 16, pk);
      }
      tmem_wait_st();
      float s0, s1, s2, s3, s4, s5, s6, s7;
      f2_unpack(acc[0], s0, s1);
      f2_unpack(acc[1], s2, s3);
      f2_unpack(acc[2], s4, s5);
      f2_unpack(acc[3], s6, s7);
      const float sum = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
      l = l * alpha + sum;
      m = m_new;
      tc_fence_before();
      // d = 64: the next S may already be there, so a fast warp could start the next tile
      // and arrive again before the slowest warp has arrived for this one; the warpgroup
      // meets here first
      if constexpr (L::RING) named_bar_sync(1 + t, BM);
      mbar_arrive(bars + 8u * (L::B_PREADY + t));
      ++nact;
      ++np;
    }

    // Epilogue: O = O_acc / l, LSE; rows with nothing kept give O = 0, LSE = -inf.
    if (nact > 0) {
      if (!bwait_warp(bars + 8u * (L::B_ODONE + t), o_par, abort_flag, to)) return;
      o_par ^= 1u;
      tc_fence_after();
    }
    const bool row_ok = i >= 0 && i < sq;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    bool staged = false;
    if constexpr (L::STAGE_O) {
     if (nact > 0) {
      staged = true;
      // This warp's 32 rows x d go through its slice of the unit's Q buffer (the unit's
      // last Q.K^T of tile t finished before O_t was signalled; a tile that computed
      // nothing never waited for its Q load, so it writes its zeros directly instead):
      // row r's 16-byte chunk c is stored at
      // chunk c ^ (r & 7) of the slice's row r, so both the row-per-lane writes and the
      // chunk-per-lane reads below touch every bank group once per 8 lanes.  The reads
      // give each store instruction 512 contiguous bytes of O (4 whole rows).
      constexpr int ROW_BYTES = D * 2, CHUNKS = ROW_BYTES / 16;
      static_assert(QT * 4 * 32 * ROW_BYTES == L::Q_BUF_BYTES, "staging slices fill one Q buffer");
      uint8_t* stage = gbase + L::OFF_Q + (k % L::QBUF) * L::Q_BUF_BYTES + (t * 4 + quarter) * (32 * ROW_BYTES);
      static_assert(D == 64, "the staged epilogue reads the whole O row at once");
      uint32_t ob[64];
      tmem_ld32x32b_x64_wait(o_addr, ob);  // the whole row of O in one load
#pragma unroll
      for (int ch = 0; ch < D / 16; ++ch) {
        uint32_t pk[8];
#pragma unroll
        for (int x = 0; x < 8; ++x)
          pk[x] = pack2<BF16>(__uint_as_float(ob[16 * ch + 2 * x]) * inv, __uint_as_float(ob[16 * ch + 2 * x + 1]) * inv);
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          const int c = 2 * ch + hc;
          *reinterpret_cast<uint4*>(stage + lane * ROW_BYTES + ((c ^ (lane & 7)) * 16)) =
              make_uint4(pk[4 * hc], pk[4 * hc + 1], pk[4 * hc + 2], pk[4 * hc + 3]);
        }
      }
      __syncwarp();
      const int row0w = rt + quarter * 32;  // this warp's first row
      uint8_t* obh = reinterpret_cast<uint8_t*>(p.o) + q_row_base(p, b, hq_t, qoff) * ROW_BYTES;
      constexpr int ROWS_PER_STORE = 32 / CHUNKS;
#pragma unroll
      for (int kk = 0; kk < 32 / ROWS_PER_STORE; ++kk) {
        const int rr = kk * ROWS_PER_STORE + lane / CHUNKS, c = lane % CHUNKS;
        const uint4 val = *reinterpret_cast<const uint4*>(stage + rr * ROW_BYTES + ((c ^ (rr & 7)) * 16));
        int orow = row0w + rr;  // the slice row's place in O
        if constexpr (MODE == MASK_CUSTOM) {
          const int blk = rr < 16 ? blk_a : blk_b;
          orow = blk >= 0 ? blk * 16 + (rr & 15) : -1;
        }
        if (orow >= 0 && orow < sq) *reinterpret_cast<uint4*>(obh + (size_t)orow * ROW_BYTES + c * 16) = val;
      }
      fence_proxy_async_smem();  // the next TMA load into this buffer comes after these accesses
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8u * (L::B_QEMPTY + (k % L::QBUF)));  // slice read back
     }
    }
    if (staged) {
    } else if (L::STAGE_SEP) {
      // Same scheme through the warp's own 4 KiB slice, one 64-column half of d per pass:
      // each store instruction then writes four whole 128-byte segments of O.
      uint8_t* stage = gbase + L::OFF_STAGE + (t * 4 + quarter) * (32 * 128);
      const int row0w = rt + quarter * 32;
      uint8_t* obase = reinterpret_cast<uint8_t*>(p.o) + (q_row_base(p, b, hq_t, qoff) + row0w) * (D * 2);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t ob[16];
          if (nact > 0) {
            tmem_ld32x32b_x16_wait(o_addr + h * 64 + ch * 16, ob);
          } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) ob[x] = 0u;
          }
          uint32_t pk[8];
#pragma unroll
          for (int x = 0; x < 8; ++x)
            pk[x] = pack2<BF16>(__uint_as_float(ob[2 * x]) * inv, __uint_as_float(ob[2 * x + 1]) * inv);
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            const int c = 2 * ch + hc;
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) * 16)) =
                make_uint4(pk[4 * hc], pk[4 * hc + 1], pk[4 * hc + 2], pk[4 * hc + 3]);
          }
        }
        __syncwarp();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int rr = kk * 4 + lane / 8, c = lane % 8;
          const uint4 val = *reinterpret_cast<const uint4*>(stage + rr * 128 + ((c ^ (rr & 7)) * 16));
          if (row0w + rr < sq) *reinterpret_cast<uint4*>(obase + rr * (D * 2) + h * 128 + c * 16) = val;
        }
        __syncwarp();  // the slice is rewritten by the next half
      }
    } else {
    OutT* orow = reinterpret_cast<OutT*>(p.o) + (q_row_base(p, b, hq_t, qoff) + (row_ok ? i : 0)) * D;
#pragma unroll
    for (int ch = 0; ch < D / 16; ++ch) {
      uint32_t ob[16];
      if (nact > 0) {
        tmem_ld32x32b_x16_wait(o_addr + ch * 16, ob);
      } else {
#pragma unroll
        for (int x = 0; x < 16; ++x) ob[x] = 0u;
      }
      uint32_t pk[8];
#pragma unroll
      for (int x = 0; x < 8; ++x)
        pk[x] = pack2<BF16>(__uint_as_float(ob[2 * x]) * inv, __uint_as_float(ob[2 * x + 1]) * inv);
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 16);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    if (L::STAGE_O && lane == 0) mbar_arrive(bars + 8u * (L::B_QEMPTY + (k % L::QBUF)));
    }
    if (row_ok && p.lse)
      p.lse[q_row_base(p, b, hq_t, qoff) + i] = l > 0.f ? (m + log2f(l)) * LN2 : -INFINITY;
    if constexpr (MODE == MASK_CUSTOM) {
      // The unit also owns the 16-row blocks of its original rows; those with nothing kept
      // were left out of the compacted list: O = 0 and LSE = -inf there, this warp's two
      // blocks written in whole 16-byte chunks by consecutive lanes.
      constexpr int ROW_BYTES = D * 2, CHUNKS = ROW_BYTES / 16;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int hb = hb0 + hh;
        if constexpr (D == 64) {
          if (hh ? live_b : live_a) continue;  // warp-uniform
        } else {
          if (hb >= p.nr16 || __ldg(p.live + (size_t)mb * p.nr16 + hb)) continue;  // warp-uniform
        }
        uint8_t* ob = reinterpret_cast<uint8_t*>(p.o) + ((size_t)(b * p.Hq + hq) * p.Sq + hb * 16) * ROW_BYTES;
#pragma unroll
        for (int q = lane; q < 16 * CHUNKS; q += 32) {
          const int rr = q / CHUNKS, c = q % CHUNKS;
          if (hb * 16 + rr < sq) *reinterpret_cast<uint4*>(ob + rr * ROW_BYTES + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (lane < 16 && hb * 16 + lane < sq && p.lse) p.lse[(size_t)(b * p.Hq + hq) * p.Sq + hb * 16 + lane] = -INFINITY;
      }
    }
  }
}

// ------------------------------------------------------------------ the kernel
template <int D, bool BF16, int MODE>
__global__ void __launch_bounds__(NTHREADS, 1) attn_fwd_kernel(const __grid_constant__ Params p) {
  using L = Layout<D, MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle needs 1024-byte tiles
  uint8_t* gbase = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = base + L::OFF_BAR;

  if (threadIdx.x == 0) {
    for (int qb2 = 0; qb2 < L::QBUF; ++qb2) {
      mbar_init(bars + 8u * (L::B_QFULL + qb2), 1);
      mbar_init(bars + 8u * (L::B_QEMPTY + qb2), L::QEMPTY_COUNT);
    }
    for (int s = 0; s < L::KSLOT; ++s) {
      mbar_init(bars + 8u * (L::B_KFULL + s), 1);
      mbar_init(bars + 8u * (L::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < L::VSLOT; ++s) {
      mbar_init(bars + 8u * (L::B_VFULL + s), 1);
      mbar_init(bars + 8u * (L::B_VEMPTY + s), 1);
    }
    for (int e = 0; e < NINFO; ++e) {
      mbar_init(bars + 8u * (L::B_IFULL + e), 1);                 // load-warp lane 0
      mbar_init(bars + 8u * (L::B_IEMPTY + e), 1 + QT * BM);      // MMA thread + softmax threads
    }
    for (int sl = 0; sl < L::S_SLOTS; ++sl) mbar_init(bars + 8u * (L::B_STILE + sl), 1);
    for (int t = 0; t < QT; ++t) {
      mbar_init(bars + 8u * (L::B_PREADY + t), BM);
      mbar_init(bars + 8u * (L::B_ODONE + t), 1);
      mbar_init(bars + 8u * (L::B_OPV + t), 1);
    }
    mbar_init(bars + 8u * L::B_DRAIN, 1);
    abort_flag[0] = 0;
    abort_flag[1] = p.status_slot;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Custom masks and variable-length work orders: the set-up above overlapped the kernels
  // that write them (dependent launch); they are read only after this point.
  if (MODE == MASK_CUSTOM || p.order) grid_dependency_wait();

  // Register rebalancing: the load / MMA warpgroup (warps 0-3) needs few registers, the
  // softmax warpgroups hold a 128-score row each.  384 x 168 = 128 x 88 + 256 x 208 exactly
  // (d = 128); 128 x 96 + 256 x 200 (d = 64).
  // Each setmaxnreg sits in the same branch as the code it budgets for.
  if (warp < 4) {
    setmaxnreg_dec<L::REGS_LOADMMA>();
    if (warp == 0) {
      load_role<D, BF16, MODE>(p, base, gbase, abort_flag, lane);
    } else if (warp == 1) {
      mma_role<D, BF16, MODE>(p, base, gbase, abort_flag, tmem, lane);
    }
  } else {
    setmaxnreg_inc<L::REGS_SOFTMAX>();
    softmax_role<D, BF16, MODE>(p, base, gbase, abort_flag, tmem, (warp - 4) >> 2, warp & 3, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && p.dynamic) {
    // this CTA takes no more units; the last CTA to get here resets the queue for the next launch
    unsigned int* q = g_sched + 2 * p.status_slot;
    __threadfence();
    if (atomicAdd(q + 1, 1u) == gridDim.x - 1) {
      __threadfence();
      atomicExch(q, 0u);
      atomicExch(q + 1, 0u);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ custom-mask pre-pass
// Bits lo .. hi-1 of a 32-bit word (clipped to the word).
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 32);
  if (hi <= lo) return 0u;
  const uint32_t upto_hi = hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  const uint32_t below_lo = (1u << lo) - 1u;
  return upto_hi & ~below_lo;
}

// One warp per (mask row block mb = batch or batch*Hq + head, 128-row query tile, 128-key
// tile).  Writes the block's kept-bit words -- the caller's bits AND the key bound
// (key < Sk) AND the band [key_lo(i), key_hi(i)) -- into a copy padded to W4 = 4 * nkt words
// per row, and a 1 into flags[(mb*nqt + qt)*nkt + kt] iff any of them is set.  The attention
// kernel then reads only these: whole word tiles by TMA, and the emptiness flags for its
// tile skipping.
__global__ void __launch_bounds__(BM) mask_prepass_kernel(const uint32_t* __restrict__ mask,
                                                          uint32_t* __restrict__ words4,
                                                          uint8_t* __restrict__ flags16, Params p,
                                                          int nmb, int write_words) {
  // One CTA per (mask row block, 128 query rows, key tile), one thread per query row: every
  // thread's four words are loaded together; each half-warp's OR is the emptiness flag of
  // one (16-row block, key tile) pair.
  grid_launch_dependents();  // the attention grid may start its set-up; it waits for our output
  const long long blk = blockIdx.x;  // grid = nmb * nqt * nkt exactly
  const int kt = (int)(blk % p.nkt);
  const long long rest = blk / p.nkt;
  const int qt = (int)(rest % p.nqt);
  const long long mbk = rest / p.nqt;
  const int W4 = 4 * p.nkt;
  int sq, sk;
  unit_lengths(p, (int)(mbk / p.mask_heads), sq, sk);
  const int off = sk - sq;
  const int i = qt * BM + (int)threadIdx.x;
  uint32_t any = 0;
  if (i < p.Sq) {
    const uint32_t* src = mask + ((size_t)mbk * p.Sq + i) * p.W;
    uint32_t* dst = words4 + ((size_t)mbk * p.Sq + i) * W4;
    // rows past the entry's length keep nothing; keys past it do not exist
    const int klo = key_lo(p, i, off);
    const int khi = i < sq ? key_hi(p, i, off, sk) : 0;  // <= sk
    uint32_t x[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int gw = kt * 4 + w;
      x[w] = gw < p.W ? __ldg(src + gw) : 0u;
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int gw = kt * 4 + w;
      x[w] &= bit_range(klo - gw * 32, khi - gw * 32);
      any |= x[w];
    }
    if (write_words) *reinterpret_cast<uint4*>(dst + kt * 4) = make_uint4(x[0], x[1], x[2], x[3]);
  }
  const uint32_t bits = __ballot_sync(0xffffffffu, any != 0u);
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r16 = qt * (BM / 16) + (int)(threadIdx.x >> 5) * 2 + h;
      if (r16 < p.nr16) flags16[((size_t)mbk * p.nr16 + r16) * p.nkt + kt] = ((bits >> (16 * h)) & 0xFFFFu) ? 1 : 0;
    }
  }
}

// Compaction of mask row block mb by the whole CTA (blockDim.x a multiple of 32, <= 1024)
// from its (16-row block, key tile) flags f [nr16][nkt] (global or shared memory): which
// 16-row blocks hold a kept entry, their ascending list (the compacted slots, -1 past its end),
// and the (compacted tile, key tile) flags as the OR over the tile's eight slots.  slot_s
// (nslots >= nqt * 8 >= nr16 ints) and live_s (nr16 bytes) are shared-memory scratch.
__device__ __forceinline__ void compact_rows(const uint8_t* f, uint8_t* __restrict__ live, int* __restrict__ rowmap,
                                             uint8_t* __restrict__ tflags, int mb, int nr16, int nkt, int nqt,
                                             int nslots, int* slot_s, uint8_t* live_s) {
  __shared__ int warp_tot[32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x, nwarp = nthr >> 5;
  for (int r = tid; r < nr16; r += nthr) {
    uint32_t any = 0;
    for (int kt = 0; kt < nkt; ++kt) any |= f[(size_t)r * nkt + kt];
    live_s[r] = any ? 1 : 0;
    live[(size_t)mb * nr16 + r] = any ? 1 : 0;
  }
  if (tid == 0) carry_s = 0;
  __syncthreads();
  // ascending list of the live blocks: a block-wide exclusive scan, nthr blocks per round
  for (int base = 0; base < nr16; base += nthr) {
    const int r = base + tid;
    const bool v = r < nr16 && live_s[r];
    const uint32_t bal = __ballot_sync(0xffffffffu, v);
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = carry_s;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (v) slot_s[before + __popc(bal & ((1u << lane) - 1u))] = r;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < nwarp; ++w) tot += warp_tot[w];
      carry_s += tot;
    }
    __syncthreads();
  }
  const int c = carry_s;
  for (int sl = tid; sl < nslots; sl += nthr) {
    if (sl >= c) slot_s[sl] = -1;
    rowmap[(size_t)mb * nslots + sl] = sl < c ? slot_s[sl] : -1;
  }
  __syncthreads();
  for (int idx = tid; idx < nqt * nkt; idx += nthr) {
    const int ct = idx / nkt, kt = idx % nkt;
    uint32_t any = 0;
    for (int sl = ct * 8; sl < ct * 8 + 8 && sl < c; ++sl) any |= f[(size_t)slot_s[sl] * nkt + kt];
    tflags[(size_t)mb * nqt * nkt + idx] = any ? 1 : 0;
  }
}

// Compaction of one mask row block (one CTA per block, 256 threads) from the pre-pass's flags.
// Shared memory: nslots (>= nqt * 8 >= nr16) slot entries and nr16 bytes of liveness.
__global__ void __launch_bounds__(256) mask_compact_kernel(const uint8_t* __restrict__ flags16,
                                                          uint8_t* __restrict__ live, int* __restrict__ rowmap,
                                                          uint8_t* __restrict__ tflags, int nr16, int nkt,
                                                          int nqt, int nslots) {
  grid_launch_dependents();  // the attention grid may start its set-up; it waits for our output
  grid_dependency_wait();    // launched as a dependent of the pre-pass: its flags are complete
  extern __shared__ int cmp_smem[];
  int* slot_s = cmp_smem;                                             // nslots
  uint8_t* live_s = reinterpret_cast<uint8_t*>(cmp_smem + nslots);    // nr16
  const int mb = blockIdx.x;
  compact_rows(flags16 + (size_t)mb * nr16 * nkt, live, rowmap, tflags, mb, nr16, nkt, nqt, nslots, slot_s, live_s);
}

// Key tiles the two Q tiles of work unit (b, any head, 256-row block qb) compute -- the same
// bounds the load warp uses (per-entry lengths, bottom-right alignment, band).
__device__ __forceinline__ int unit_weight(const Params& p, int b, int qb) {
  int sq, sk, qoff, koff;
  unit_span(p, b, sq, sk, qoff, koff);
  const int off = sk - sq;
  int w = 0;
#pragma unroll
  for (int t = 0; t < QT; ++t) {
    const int r0 = qb * UNIT_ROWS + (p.pair ? 0 : t * BM);
    const int r1 = min(r0 + BM - 1, sq - 1);
    const int rf = p.er >= 0 ? max(r0, -off - p.er) : r0;
    const int klo = key_lo(p, rf, off), khi = key_hi(p, r1, off, sk);
    if (r0 < sq && rf <= r1 && khi > klo) w += (khi - 1) / BN - klo / BN + 1;
  }
  return w;
}

// Work order of a variable-length batch (one CTA): the (batch entry, 256-row block) pairs
// sorted by the key tiles they compute, most first (a counting sort over the weights
// 0 .. 2 * nkt), so the work queue hands out the longest units first whatever the entries'
// lengths.  Pairs of equal weight come in no particular order (each unit's result does not
// depend on when it runs).  Shared memory: nbins = 2 * nkt + 1 counters.
constexpr int ORDER_THREADS = 1024;
__global__ void __launch_bounds__(ORDER_THREADS) unit_order_kernel(const Params p, int* __restrict__ order) {
  grid_launch_dependents();  // the attention grid may start its set-up; it waits for our output
  extern __shared__ int bins[];
  const int tid = threadIdx.x, lane = tid & 31;
  const int nbins = 2 * p.nkt + 1, npairs = p.B * p.nqb;
  for (int i = tid; i < nbins; i += ORDER_THREADS) bins[i] = 0;
  __syncthreads();
  for (int pr = tid; pr < npairs; pr += ORDER_THREADS) {
    const int b = pr / p.nqb;
    atomicAdd(&bins[nbins - 1 - unit_weight(p, b, pr - b * p.nqb)], 1);
  }
  __syncthreads();
  if (tid < 32) {
    // exclusive scan of the bins by one warp: each lane a contiguous chunk, then the lanes'
    // totals scanned with shuffles
    const int per = (nbins + 31) / 32, lo = lane * per, hi = min(lo + per, nbins);
    int tot = 0;
    for (int i = lo; i < hi; ++i) tot += bins[i];
    int incl = tot;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    int run = incl - tot;
    for (int i = lo; i < hi; ++i) {
      const int c = bins[i];
      bins[i] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int pr = tid; pr < npairs; pr += ORDER_THREADS) {
    const int b = pr / p.nqb;
    order[atomicAdd(&bins[nbins - 1 - unit_weight(p, b, pr - b * p.nqb)], 1)] = pr;
  }
}

}  // namespace attn

// ====================================================================== host side
namespace attn {
namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_inject{0};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

struct DeviceInfo {
  int state = 0;  // 0 unknown, 1 usable, -1 not an sm_103 device
  int sms = 0;
};
std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

int device_info(int& sms, int& dev) {
  dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  DeviceInfo& di = g_dev[dev];
  if (di.state == 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_DEVICE;
    di.state = (major == 10 && minor == 3) ? 1 : -1;
    di.sms = n;
  }
  if (di.state != 1) return ATTN_ERR_DEVICE;
  sms = di.sms;
  return ATTN_OK;
}

// Host-side counters (attn_debug_counters): workspace allocations, tensor-map encodes and
// tensor-map cache hits since the library was loaded.
std::atomic<unsigned long long> g_ws_allocs{0}, g_map_encodes{0}, g_map_hits{0};

// Tensor maps cached by (kind, address, dims, box rows): a map holds nothing but these, so a
// cached map is valid for any later call that names the same buffer with the same shape.
// Least-recently-used replacement over a small table.
enum MapKind { MAP_F16 = 0, MAP_BF16 = 1, MAP_WORDS = 2 };
struct MapKey {
  int kind;
  const void* ptr;
  long long d0, d1, d2;
  int box_rows;
  bool operator==(const MapKey& o) const {
    return kind == o.kind && ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && box_rows == o.box_rows;
  }
};
constexpr int MAP_CACHE = 64;
struct MapSlot {
  MapKey key;
  CUtensorMap map;
  unsigned long long used = 0;  // 0 = empty
};
std::mutex g_map_mutex;
MapSlot g_maps[MAP_CACHE];
unsigned long long g_map_clock = 0;

template <class Encode>
int cached_map(CUtensorMap* m, const MapKey& key, Encode encode) {
  {
    std::lock_guard<std::mutex> lk(g_map_mutex);
    for (MapSlot& e : g_maps)
      if (e.used && e.key == key) {
        e.used = ++g_map_clock;
        *m = e.map;
        g_map_hits.fetch_add(1);
        return ATTN_OK;
      }
  }
  const int rc = encode(m);
  if (rc != ATTN_OK) return rc;
  g_map_encodes.fetch_add(1);
  std::lock_guard<std::mutex> lk(g_map_mutex);
  MapSlot* victim = &g_maps[0];
  for (MapSlot& e : g_maps)
    if (e.used < victim->used) victim = &e;
  victim->key = key;
  victim->map = *m;
  victim->used = ++g_map_clock;
  return ATTN_OK;
}

// [rows = B*H][S][d] tensor as a 3-D map {d, S, B*H}; box {64, box_rows, 1}: one 128-byte
// swizzle span of box_rows rows.  Rows past S read as zeros.
int encode_map(CUtensorMap* m, const void* ptr, bool bf16, int d, int S, long long BH, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return ATTN_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

int make_map(CUtensorMap* m, const void* ptr, bool bf16, int d, int S, long long BH, int box_rows = 128) {
  return cached_map(m, MapKey{bf16 ? MAP_BF16 : MAP_F16, ptr, d, S, BH, box_rows},
                    [&](CUtensorMap* out) { return encode_map(out, ptr, bf16, d, S, BH, box_rows); });
}

// Kept-bit words of a custom mask after the pre-pass: 3-D map {W4, S, nmb} of uint32, box
// {4 words, box_rows, 1}: one key tile's words for one 16-row block (gathered per slot) or
// for the 256 rows of a unit whose compacted slots are its own rows.
int encode_mask_map(CUtensorMap* m, const uint32_t* words4, int W4, int Sq, int nmb, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return ATTN_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)W4, (cuuint64_t)Sq, (cuuint64_t)nmb};
  cuuint64_t strides[2] = {(cuuint64_t)W4 * 4, (cuuint64_t)Sq * (cuuint64_t)W4 * 4};
  cuuint32_t box[3] = {BN / 32, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(words4), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

int make_mask_map(CUtensorMap* m, const uint32_t* words4, int W4, int Sq, int nmb, int box_rows) {
  return cached_map(m, MapKey{MAP_WORDS, words4, W4, Sq, nmb, box_rows},
                    [&](CUtensorMap* out) { return encode_mask_map(out, words4, W4, Sq, nmb, box_rows); });
}

// ---------------------------------------------------------------- per-stream state
// Every (device, stream) the library launches on gets a status slot (the index of its word
// in g_attn_status; slot 0 is shared by the streams beyond the table) and, once it runs a
// custom mask, a workspace for the mask kernels: a stream-ordered allocation that is reused
// by every later call on that stream and replaced (the old block freed in stream order) only
// when a call needs more.  `m` is held while a call enqueues work that uses the workspace, so
// no call frees a block another call on the same stream has already handed to a kernel.
struct StreamKey {
  int dev;
  void* stream;
  bool operator==(const StreamKey& o) const { return dev == o.dev && stream == o.stream; }
};
struct StreamKeyHash {
  size_t operator()(const StreamKey& k) const {
    return std::hash<void*>()(k.stream) ^ (std::hash<int>()(k.dev) * 0x9E3779B97F4A7C15ull);
  }
};
struct StreamState {
  int slot = 0;
  std::mutex m;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};
std::mutex g_streams_mutex;
std::unordered_map<StreamKey, std::unique_ptr<StreamState>, StreamKeyHash> g_streams;
int g_next_slot[64];

// The state of (dev, stream), created on first use when `create`; nullptr if absent.
StreamState* stream_state(int dev, void* stream, bool create) {
  std::lock_guard<std::mutex> lk(g_streams_mutex);
  const StreamKey key{dev, stream};
  auto it = g_streams.find(key);
  if (it != g_streams.end()) return it->second.get();
  if (!create) return nullptr;
  auto st = std::make_unique<StreamState>();
  int& next = g_next_slot[dev];
  if (next == 0) next = 1;
  st->slot = next < STATUS_SLOTS ? next++ : 0;
  StreamState* raw = st.get();
  g_streams.emplace(key, std::move(st));
  return raw;
}

// Makes s.ws hold at least `need` bytes (caller holds s.m).  Grows in whole MiB.
int ensure_workspace(StreamState& s, size_t need, cudaStream_t st) {
  if (s.ws_bytes >= need) return ATTN_OK;
  const size_t bytes = (need + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
  if (s.ws) {
    if (cudaFreeAsync(s.ws, st) != cudaSuccess) return ATTN_ERR_CUDA;
    s.ws = nullptr;
    s.ws_bytes = 0;
  }
  void* p = nullptr;
  if (cudaMallocAsync(&p, bytes, st) != cudaSuccess) return ATTN_ERR_CUDA;
  g_ws_allocs.fetch_add(1);
  s.ws = p;
  s.ws_bytes = bytes;
  return ATTN_OK;
}

// Scratch of the custom-mask kernels for nmb mask row blocks (B, or B*Hq for per-head masks).
struct MaskScratch {
  // kept-bit words [nmb][Sq][W4], flags per (16-row block, key tile) [nmb][nr16][nkt],
  // live 16-row blocks [nmb][nr16], compacted slot -> block [nmb][nqb * 16] (int, 16 slots per
  // 256-row work unit), compacted tile flags [nmb][nqt][nkt]; every part starts on a 256-byte
  // boundary
  size_t off_flags16, off_live, off_rowmap, off_tflags, bytes;
  static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
  MaskScratch(long long nmb, int Sq, int Sk) {
    const long long nqt = (Sq + BM - 1) / BM, nkt = (Sk + BN - 1) / BN, nr16 = (Sq + 15) / 16;
    const long long nslots = (Sq + UNIT_ROWS - 1) / UNIT_ROWS * 16;
    off_flags16 = round256((size_t)nmb * Sq * (size_t)(4 * nkt) * 4);
    off_live = off_flags16 + round256((size_t)(nmb * nr16 * nkt));
    off_rowmap = off_live + round256((size_t)(nmb * nr16));
    off_tflags = off_rowmap + round256((size_t)(nmb * nslots) * 4);
    bytes = off_tflags + round256((size_t)(nmb * nqt * nkt));
  }
  size_t total() const { return bytes; }
};

// Runs the mask pre-pass into `scratch` (MaskScratch layout) and points p at its output.
int prepare_mask(Params& p, const uint32_t* mask_bits, void* scratch, cudaStream_t st, int dev) {
  const int nmb = p.B * p.mask_heads;
  const MaskScratch ms(nmb, p.Sq, p.Sk);
  uint8_t* base = reinterpret_cast<uint8_t*>(scratch);
  uint32_t* words4 = reinterpret_cast<uint32_t*>(base);
  uint8_t* flags16 = base + ms.off_flags16;
  uint8_t* live = base + ms.off_live;
  int* rowmap = reinterpret_cast<int*>(base + ms.off_rowmap);
  uint8_t* tflags = base + ms.off_tflags;
  const long long blocks = (long long)nmb * p.nqt * p.nkt;
  if (blocks > INT_MAX) return ATTN_ERR_INVALID;
  const int nslots = p.nqb * 16;
  p.tflags = tflags;
  p.rowmap = rowmap;
  p.live = live;
  const size_t cmp_smem = (size_t)nslots * 4 + (size_t)p.nr16;
  if (cmp_smem > 227 * 1024) return ATTN_ERR_UNSUPPORTED;
  if (cmp_smem > 48 * 1024) {
    static std::atomic<unsigned long long> attr_set{0};  // bit per device
    const unsigned long long bit = 1ull << dev;
    if (!(attr_set.load() & bit)) {
      if (cudaFuncSetAttribute(mask_compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
          cudaSuccess)
        return ATTN_ERR_CUDA;
      attr_set.fetch_or(bit);
    }
  }
  // When no bound applies (no band or causal bound, no per-entry lengths) and the key count is
  // a multiple of the key tile, the padded words equal the caller's words byte for byte: the
  // kernel then reads those (through 16-byte-aligned rows), and the pre-pass only flags.
  const bool words_in_place = p.Sk % BN == 0 && p.W == 4 * p.nkt && p.wl < 0 && p.er < 0 && !p.lens_q &&
                              !p.lens_k && !p.cu_q && (reinterpret_cast<uintptr_t>(mask_bits) & 15u) == 0;
  mask_prepass_kernel<<<(unsigned)blocks, BM, 0, st>>>(mask_bits, words4, flags16, p, nmb, words_in_place ? 0 : 1);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nmb);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = cmp_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mask_compact_kernel, (const uint8_t*)flags16, live, rowmap, tflags, p.nr16, p.nkt,
                           p.nqt, nslots) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  const uint32_t* words = words_in_place ? mask_bits : words4;
  int rc = make_mask_map(&p.tm_m, words, 4 * p.nkt, p.Sq, nmb, 16);
  return rc != ATTN_OK ? rc : make_mask_map(&p.tm_m256, words, 4 * p.nkt, p.Sq, nmb, UNIT_ROWS);
}

template <int D, bool BF16, int MODE>
int launch(const Params& p, int grid, cudaStream_t st, int dev, bool dependent) {
  using L = Layout<D, MODE>;
  auto kern = attn_fwd_kernel<D, BF16, MODE>;
  static std::atomic<unsigned long long> attr_set{0};  // bit per device
  const unsigned long long bit = 1ull << dev;
  if (!(attr_set.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_ALLOC) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_set.fetch_or(bit);
  }
  if (dependent) {
    // Launched as a programmatic dependent of the kernel just enqueued on `st` (the mask
    // compaction or the work order), whose output it waits for with griddepcontrol.wait.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = L::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  kern<<<grid, NTHREADS, L::SMEM_ALLOC, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D, bool BF16>
int launch_mode(const Params& p, int mode, int grid, cudaStream_t st, int dev, bool dependent) {
  switch (mode) {
    case MASK_NONE: return launch<D, BF16, MASK_NONE>(p, grid, st, dev, dependent);
    case MASK_CAUSAL: return launch<D, BF16, MASK_CAUSAL>(p, grid, st, dev, dependent);
    case MASK_BAND: return launch<D, BF16, MASK_BAND>(p, grid, st, dev, dependent);
    default: return launch<D, BF16, MASK_CUSTOM>(p, grid, st, dev, dependent);
  }
}

// ---------------------------------------------------------------- no-allocation variant
// Scratch for attn_fwd_noalloc: a fixed device array instead of a stream-ordered workspace.
// In host code the symbol is only a host-side stand-in; its device address comes from
// cudaGetSymbolAddress, asked for on every call with the caller's device current, so a
// context that was reset or replaced (the module then reloads, possibly elsewhere) never
// gets a stale address.  The first call on a device loads the module's device code.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

int noalloc_scratch_address(void** out) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
  *out = ptr;
  return ATTN_OK;
}

int fwd_impl(const attn_fwd_params_t& a, bool noalloc = false) {
  // ---- validation (no CUDA call before this block is passed)
  if (!a.q || !a.k || !a.v || !a.o) return ATTN_ERR_INVALID;
  const bool packed = a.cu_seqlens_q != nullptr;
  if (packed != (a.cu_seqlens_k != nullptr)) return ATTN_ERR_INVALID;
  if (packed && (a.seqlens_q || a.seqlens_k || a.max_seqlen_q < 1 || a.max_seqlen_k < 1)) return ATTN_ERR_INVALID;
  if (packed && a.mask_bits) return ATTN_ERR_UNSUPPORTED;
  if (a.B < 1 || a.Hq < 1 || a.Hkv < 1 || a.Sq < 1 || a.Sk < 1 || (!packed && a.Sk < a.Sq) ||
      a.Hq % a.Hkv != 0)
    return ATTN_ERR_INVALID;
  if (a.window_left < -1 || a.window_right < -1) return ATTN_ERR_INVALID;
  if (a.mask_per_head != 0 && a.mask_per_head != 1) return ATTN_ERR_INVALID;
  if (a.d != 64 && a.d != 128) return ATTN_ERR_UNSUPPORTED;
  if (a.dtype != ATTN_F16 && a.dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (!(a.scale > 0.f) || !std::isfinite(a.scale)) return ATTN_ERR_INVALID;
  const uintptr_t a16 = (uintptr_t)a.q | (uintptr_t)a.k | (uintptr_t)a.v | (uintptr_t)a.o;
  if (a16 & 15u) return ATTN_ERR_INVALID;
  if (((uintptr_t)a.lse & 3u) || ((uintptr_t)a.mask_bits & 3u) || ((uintptr_t)a.seqlens_q & 3u) ||
      ((uintptr_t)a.seqlens_k & 3u) || ((uintptr_t)a.cu_seqlens_q & 3u) || ((uintptr_t)a.cu_seqlens_k & 3u))
    return ATTN_ERR_INVALID;
  // the per-entry extents the kernel works with (packed: the longest entry's)
  const int Sq = packed ? a.max_seqlen_q : a.Sq, Sk = packed ? a.max_seqlen_k : a.Sk;
  const long long nqb = (Sq + UNIT_ROWS - 1) / UNIT_ROWS;
  if ((long long)a.B * a.Hq * Sk > INT_MAX || (long long)a.B * a.Hq * nqb > INT_MAX ||
      (long long)a.Hq * a.Sq > INT_MAX || (long long)a.Hkv * a.Sk > INT_MAX)
    return ATTN_ERR_INVALID;

  int sms = 0, dev = 0;
  int rc = device_info(sms, dev);
  if (rc != ATTN_OK) return rc;

  Params p;
  std::memset(&p, 0, sizeof p);
  const bool bf16 = a.dtype == ATTN_BF16;
  // padded: {d, Sq, B*Hq}; packed: {d, total rows, Hq} (an entry's rows at its offset)
  const long long qz = packed ? a.Hq : (long long)a.B * a.Hq, kz = packed ? a.Hkv : (long long)a.B * a.Hkv;
  if ((rc = make_map(&p.tm_q, a.q, bf16, a.d, a.Sq, qz)) != ATTN_OK) return rc;
  if ((rc = make_map(&p.tm_k, a.k, bf16, a.d, a.Sk, kz)) != ATTN_OK) return rc;
  if ((rc = make_map(&p.tm_v, a.v, bf16, a.d, a.Sk, kz)) != ATTN_OK) return rc;
  if (a.mask_bits && (rc = make_map(&p.tm_q16, a.q, bf16, a.d, a.Sq, (long long)a.B * a.Hq, 16)) != ATTN_OK)
    return rc;
  p.o = a.o;
  p.lse = a.lse;
  p.visited = a.visited;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.cu_q = a.cu_seqlens_q;
  p.cu_k = a.cu_seqlens_k;
  p.q_rows = a.Sq;
  p.k_rows = a.Sk;
  p.g = a.Hq / a.Hkv;
  p.nqb = (int)nqb;
  p.nkt = (Sk + BN - 1) / BN;
  p.nqt = (Sq + BM - 1) / BM;
  p.nr16 = (Sq + 15) / 16;
  p.W = (Sk + 31) / 32;
  p.num_units = a.B * a.Hq * (int)nqb;
  // GQA head pairs when one Q tile holds a whole entry's queries (no custom mask: its
  // compaction works on the rows of one head)
  p.pair = (Sq <= BM && (a.Hq / a.Hkv) % 2 == 0 && !a.mask_bits) ? 1 : 0;
  if (p.pair) p.num_units = a.B * (a.Hq / 2);
  p.wl = a.window_left;
  p.er = a.causal ? 0 : a.window_right;  // causal: nothing right of the aligned position
  p.mask_heads = (a.mask_bits && a.mask_per_head) ? a.Hq : 1;
  p.lens_q = a.seqlens_q;
  p.lens_k = a.seqlens_k;
  p.causal = (p.er >= 0 && p.wl < 0) ? 1 : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  {
    const unsigned long long us = (g_timeout_ns.load() + 999ull) / 1000ull;
    p.timeout_us = us > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)us;
  }
  p.inject = g_inject.exchange(0);
  const int grid = p.num_units < sms ? p.num_units : sms;
  const int mode = a.mask_bits                        ? MASK_CUSTOM
                   : (p.wl < 0 && p.er < 0)            ? MASK_NONE
                   : (p.wl < 0 && p.er == 0)           ? MASK_CAUSAL
                                                       : MASK_BAND;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(a.stream);
  // The stream's status slot.  attn_fwd_noalloc allocates nothing, not even the host-side
  // entry of a stream it has not seen: such a stream reports through the shared slot 0.
  StreamState* ss = stream_state(dev, a.stream, !noalloc);
  p.status_slot = ss ? ss->slot : 0;
  // Without a custom mask, units with no right bound on the keys, causal units (longest
  // first), windows of at least 1024 keys and variable-length batches are taken from the
  // stream's work queue, so CTAs that finish early take more.
  // Custom-mask units and narrower windows (a few key tiles per unit) keep the fixed snake
  // walk over the longest-first order, which balanced them better (measured).  The shared
  // slot 0 may serve launches on several streams at once, so those keep the fixed walk too.
  const bool varlen_batch = packed || a.seqlens_q || a.seqlens_k;
  const bool wide = p.wl < 0 || p.wl >= 1024;
  p.dynamic = (p.status_slot != 0 && (varlen_batch || (!a.mask_bits && (p.er < 0 || (p.er == 0 && wide))))) ? 1 : 0;
  // Variable-length batches with the work queue get a work order, longest units first.
  const bool with_order = varlen_batch && p.dynamic && 2ll * p.nkt + 1 <= 8192;
  const bool custom = mode == MASK_CUSTOM;
  const auto run = [&]() {
    const bool dep = custom || with_order;
    if (a.d == 64)
      return bf16 ? launch_mode<64, true>(p, mode, grid, st, dev, dep) : launch_mode<64, false>(p, mode, grid, st, dev, dep);
    return bf16 ? launch_mode<128, true>(p, mode, grid, st, dev, dep)
                : launch_mode<128, false>(p, mode, grid, st, dev, dep);
  };
  if (!custom && !with_order) return run();
  // Scratch in the stream's workspace: the mask kernels' output, then the work order.
  const size_t mask_bytes = custom ? MaskScratch((long long)a.B * p.mask_heads, a.Sq, a.Sk).total() : 0;
  const size_t order_off = (mask_bytes + 255) & ~(size_t)255;
  const size_t need = order_off + (with_order ? (size_t)a.B * p.nqb * sizeof(int) : 0);
  if (noalloc) {
    // the fixed array (attn_fwd_noalloc takes no variable lengths): reject what does not fit
    // before anything is launched
    if (need > (size_t)ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_INVALID;
    void* scratch = nullptr;
    if ((rc = noalloc_scratch_address(&scratch)) != ATTN_OK) return rc;
    if ((rc = prepare_mask(p, a.mask_bits, scratch, st, dev)) != ATTN_OK) return rc;
    return run();
  }
  std::lock_guard<std::mutex> lk(ss->m);
  if ((rc = ensure_workspace(*ss, need, st)) != ATTN_OK) return rc;
  if (with_order) {
    // first, as a plain launch: the mask kernels (if any) start after it has finished
    int* order = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ss->ws) + order_off);
    unit_order_kernel<<<1, ORDER_THREADS, (2 * p.nkt + 1) * sizeof(int), st>>>(p, order);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    p.order = order;
  }
  if (custom && (rc = prepare_mask(p, a.mask_bits, ss->ws, st, dev)) != ATTN_OK) return rc;
  return run();
}

attn_fwd_params_t square_params(const void* q, const void* k, const void* v, void* o, float* lse,
                                const uint32_t* mask_bits, int B, int Hq, int Hkv, int S, int d,
                                int causal, float scale, int dtype, void* stream, uint8_t* visited) {
  attn_fwd_params_t a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.mask_bits = mask_bits;
  a.mask_per_head = 0;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = S;
  a.Sk = S;
  a.d = d;
  a.causal = causal;
  a.window_left = -1;
  a.window_right = -1;
  a.scale = scale;
  a.dtype = dtype;
  a.stream = stream;
  a.visited = visited;
  return a;
}

}  // namespace
}  // namespace attn

// ====================================================================== C-ABI
extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             const uint32_t* mask_bits, int B, int Hq, int Hkv, int S, int d, int causal,
             float scale, int dtype, void* stream) {
  return attn::fwd_impl(attn::square_params(q, k, v, o, lse, mask_bits, B, Hq, Hkv, S, d, causal,
                                            scale, dtype, stream, nullptr));
}

int attn_fwd_ex(const attn_fwd_params_t* params) {
  if (!params) return ATTN_ERR_INVALID;
  return attn::fwd_impl(*params);
}

int attn_fwd_visited(const void* q, const void* k, const void* v, void* o, float* lse,
                     const uint32_t* mask_bits, int B, int Hq, int Hkv, int S, int d, int causal,
                     float scale, int dtype, void* stream, uint8_t* visited) {
  if (!visited) return ATTN_ERR_INVALID;
  return attn::fwd_impl(attn::square_params(q, k, v, o, lse, mask_bits, B, Hq, Hkv, S, d, causal,
                                            scale, dtype, stream, visited));
}

int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                     const uint32_t* mask_bits, int B, int Hq, int Hkv, int S, int d, int causal,
                     float scale, int dtype, void* stream) {
  return attn::fwd_impl(attn::square_params(q, k, v, o, lse, mask_bits, B, Hq, Hkv, S, d, causal,
                                            scale, dtype, stream, nullptr),
                        true);
}

int attn_check(void* stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_DEVICE;
  const attn::StreamState* ss = attn::stream_state(dev, stream, false);
  const size_t off = (size_t)(ss ? ss->slot : 0) * sizeof(unsigned int);
  // The status word is read in stream order, after everything enqueued on `stream` so far.
  unsigned int status = 0;
  if (cudaMemcpyFromSymbolAsync(&status, g_attn_status, sizeof status, off, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (status != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_attn_status, &zero, sizeof zero, off, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

int attn_release_workspace(void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_DEVICE;
  attn::StreamState* ss = attn::stream_state(dev, stream, false);
  if (!ss) return ATTN_OK;
  std::lock_guard<std::mutex> lk(ss->m);
  if (ss->ws) {
    if (cudaFreeAsync(ss->ws, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    ss->ws = nullptr;
    ss->ws_bytes = 0;
  }
  return ATTN_OK;
}

int attn_debug_counters(unsigned long long* out, int n) {
  if (!out || n < 1) return ATTN_ERR_INVALID;
  const unsigned long long v[3] = {attn::g_ws_allocs.load(), attn::g_map_encodes.load(), attn::g_map_hits.load()};
  for (int i = 0; i < n; ++i) out[i] = i < 3 ? v[i] : 0ull;
  return ATTN_OK;
}

const char* attn_strerror(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dim or dtype";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case ATTN_ERR_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

int attn_tile_shape(int d, int* bm, int* bn) {
  if (!bm || !bn) return ATTN_ERR_INVALID;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  *bm = attn::BM;
  *bn = attn::BN;
  return ATTN_OK;
}

int attn_set_wait_timeout_ns(unsigned long long ns) {
  attn::g_timeout_ns.store(ns ? ns : attn::kDefaultTimeoutNs);
  return ATTN_OK;
}

int attn_debug_inject(int flag) {
  if (flag != 0 && flag != 1) return ATTN_ERR_INVALID;
  attn::g_inject.store(flag);
  return ATTN_OK;
}

int attn_version(void) { return 100; }

}  // extern "C"
