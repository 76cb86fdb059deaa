// fa_fwd_kernel.cuh — the sm_103a attention-forward kernel.
//
// Computes, per (batch b, head h, query row i):
//   t_ij = log2(e) * (scale * q_i . k_j + mask[b, j])       (log2-domain scores)
//   O_i  = sum_j 2^(t_ij - m_i) v_j / sum_j 2^(t_ij - m_i),  LSE_i = ln2 * (m_i + log2 l_i)
// FlashAttention-style: the key axis is walked in 128-key blocks with a
// running row max m, running denominator l and a rescaled accumulator O
// ("算子加速：注意力、编译与融合", section "注意力：从O(N²)显存到分块": the figure and
// the `blocked` example's m / l / acc recurrence), so the score matrix never
// leaves the SM.  exp is taken as exp2 with log2(e) folded into the scale.
//
// One persistent CTA per SM walks work units (b·h, 256 query rows = two
// 128-row query tiles).  Warp roles (384 threads):
//   warps 0-3  softmax warpgroup for query tile 0 (one thread per row)
//   warps 4-7  softmax warpgroup for query tile 1
//   warp  8    TMA producer: Q tiles, then K_j, V_j into a shared-memory ring
//   warp  9    MMA issuer and TMEM owner (the warp runs the loop, one elected
//              lane issues each MMA batch and commit); at D <= 64 tile 0's
//              MMAs only
//   warp  10   staged fp32 mask: the mask copier (TMA); otherwise idle
//   warp  11   D <= 64: tile 1's MMA issuer; otherwise idle
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D),
// O1 [256+D, 256+2D).  At D = 128 P (bf16) is written over the first 64
// columns of its S block; at D <= 64 P0 and P1 have 64 columns of their own
// after O1, so the next S can be computed while P waits for its P·V.  P is
// fed to the P·V MMA straight from tensor memory.
//
// Every mbarrier wait is bounded in time: past the limit the CTA records
// FA_ERR_TIMEOUT in a device status word, drains its own in-flight copies and
// MMAs, frees tensor memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <climits>
#include <cstdint>

#include "fa_fastdiv.h"
#include "fa_window_geom.h"
#include "sm100_ptx.cuh"

namespace fa {

constexpr int kStatusTimeout = 4;     // == FA_ERR_TIMEOUT
constexpr int kStatusDebugCheck = 5;  // == FA_ERR_DEBUG_CHECK
constexpr uint32_t kSuspendNs = 20000;  // longest sleep inside one mbarrier poll


// How the general softmax path reads additive mask values, one kind per
// launch (chosen on the host from the mask, Nk and the alignment):
//   none          only the key-range checks;
//   key fp32 x4   a key-padding mask [B][Nk] (one row shared by every query
//                 row of a batch entry) with Nk a multiple of 4: each lane
//                 loads 4 of a key block's 128 values before S is ready, and
//                 the general path takes them from the lanes by shuffles;
//   fp32 / u8     one element per load (rows not 16-byte aligned, or a
//                 key-padding mask with Nk not a multiple of 4);
//   u8 x16        a per-(query, key) byte mask, 16 bytes per load;
//   fp32 staged   a per-(query, key) fp32 mask whose rows are 16-byte
//                 multiples, copied by TMA into shared memory in 16 KB pieces
//                 of 128 rows x 32 keys by a producer warp, ahead of the
//                 softmax.
enum : int {
  kMaskNone = 0,
  kMaskF32Vec = 1,  // key fp32 x4
  kMaskF32Scalar = 2,
  kMaskU8Vec = 3,
  kMaskU8Scalar = 4,
  kMaskF32Staged = 5,
};
// Deepest K/V ring (barrier pairs reserved).
constexpr int kMaxStages = 16;
// Staged mask ring: slots of 16 KB (128 rows x 128 bytes) and the full
// barriers that signal them (two per slot; the reason is given in Cfg).
constexpr int kMaskSlots = 4;
constexpr int kMaskFullBars = 2 * kMaskSlots;

// F8: Q and K are e4m3 (one byte) with per-128-row block scales and
// S = Q K^T runs as kind::f8f6f4 MMAs; V and P stay bf16.  MK: mask kind
// (the staged kind takes shared memory from the K/V ring).
template <int D, bool F8 = false, int MK = kMaskNone>
struct Cfg {
  static_assert(D == 32 || D == 64 || D == 128, "head dim");
  static constexpr int BM = 128;                       // query rows per tile
  static constexpr int BN = 128;                       // keys per tile
  // bf16 tiles (V always; Q and K without F8)
  static constexpr int SW = (D >= 64) ? 128 : 64;      // swizzle span = bytes per chunk row
  static constexpr int CHUNK_ELEMS = SW / 2;           // bf16 per chunk row
  static constexpr int NCHUNK = D / CHUNK_ELEMS;       // chunks across the head dim
  static constexpr int CHUNK_BYTES = BN * SW;          // one 128-row chunk
  static constexpr int TILE_BYTES = BN * D * 2;        // one 128-row bf16 tile = one ring stage
  // Q and K tiles (operands of S = Q K^T)
  static constexpr int QK_ELEM = F8 ? 1 : 2;
  static constexpr int QK_SW = F8 ? D : SW;            // fp8 rows are D bytes: 128/64/32-byte swizzle
  static constexpr int QK_CHUNK_ELEMS = QK_SW / QK_ELEM;
  static constexpr int QK_NCHUNK = D / QK_CHUNK_ELEMS;
  static constexpr int QK_CHUNK_BYTES = BN * QK_SW;
  static constexpr int QK_TILE_BYTES = BN * D * QK_ELEM;
  static constexpr int QK_SBO = 8 * QK_SW;
  static constexpr uint32_t QK_LAYOUT = QK_SW == 128 ? 2u : (QK_SW == 64 ? 4u : 6u);
  static constexpr int QK_KSTEP = F8 ? 32 : 16;        // K elements per MMA instruction
  static constexpr int S_MMAS = D / QK_KSTEP;          // MMA instructions per S tile
  // Start-address offset (16-byte units) of k-step kk of S = Q K^T: each
  // k-step covers 32 bytes of a row (16 bf16 or 32 e4m3).
  __host__ __device__ static constexpr uint32_t s_off(int kk) {
    return ((kk / (QK_CHUNK_ELEMS / QK_KSTEP)) * QK_CHUNK_BYTES +
            (kk % (QK_CHUNK_ELEMS / QK_KSTEP)) * 32) >> 4;
  }
#ifndef FA_STAGES_D128
#define FA_STAGES_D128 5
#endif
#ifndef FA_STAGES_D64
#define FA_STAGES_D64 6
#endif
#ifndef FA_STAGES_D32
#define FA_STAGES_D32 8
#endif
  // Staged mask pieces: 16 KB each (128 rows x 32 fp32 keys, 128-byte
  // swizzle), a ring of MASK_SLOTS, MASK_PIECES per 128-key block per query
  // tile.
  static constexpr bool STAGED_MASK = MK == kMaskF32Staged;
  static constexpr int MASK_SLOTS = kMaskSlots;
  // Piece i lands on full barrier i mod MASK_FULL_BARS.  The two warpgroups
  // take pieces alternately (a block's pieces for tile 0, then for tile 1),
  // so a warp may wait for a piece up to 2 * MASK_PIECES - 1 pieces ahead of
  // the oldest one not yet consumed; with one barrier per slot that wait could
  // be two phases ahead of the barrier and its parity test would pass at
  // once.  Two barriers per slot keep every wait within one phase.
  static constexpr int MASK_FULL_BARS = kMaskFullBars;
  static constexpr int MASK_PIECE_BYTES = 128 * 128;
  static constexpr int MASK_PIECE_KEYS = 32;
  static constexpr int MASK_PIECES = 128 / MASK_PIECE_KEYS;
  // K/V ring depth (build options FA_STAGES_D*): at D = 128 as deep as
  // shared memory allows (227 KB per CTA); at D <= 64 deeper rings (up to
  // 12 / 16 stages fit) measured no faster than 6 / 8.
  static constexpr int STAGES = STAGED_MASK ? ((D == 128) ? 3 : (D == 64 ? 6 : 16))
                                            : ((D == 128) ? (F8 ? 6 : FA_STAGES_D128)
                                                          : (D == 64 ? FA_STAGES_D64 : FA_STAGES_D32));
  static_assert(STAGES <= kMaxStages, "ring barriers");
  static constexpr int SMEM_Q = 2 * QK_TILE_BYTES;
  static constexpr int SMEM_MASK = STAGED_MASK ? MASK_SLOTS * MASK_PIECE_BYTES : 0;
  static constexpr int SMEM_RING = STAGES * TILE_BYTES;
  // D <= 64: each softmax warp stages its 32 output rows here for coalesced
  // stores (at D = 128 shared memory is full; the epilogue shuffles).
  static constexpr bool EPI_SMEM = D <= 64;
  static constexpr int EPI_WARP_BYTES = 32 * D * 2;
  static constexpr int SMEM_EPI = EPI_SMEM ? 8 * EPI_WARP_BYTES : 0;
  static constexpr int SMEM_BAR = 1024;
  static constexpr int SMEM_USED =
      1024 /*align slack*/ + SMEM_Q + SMEM_MASK + SMEM_RING + SMEM_EPI + SMEM_BAR;
  // 512 TMEM columns per CTA => one CTA per SM; pad shared memory so that a
  // second CTA never lands on the SM and blocks in tcgen05.alloc.
  static constexpr int SMEM_BYTES = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static constexpr int SBO = 8 * SW;                   // bytes between 8-row core-matrix groups
  static constexpr uint32_t LAYOUT = (SW == 128) ? 2u : 4u;  // UMMA SWIZZLE_128B / SWIZZLE_64B
  static constexpr int TMEM_COLS = 512;
  static constexpr int COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
  // At D <= 64 the bf16 P of each tile (64 columns) has columns of its own,
  // so S_t(j+1) can be computed while P_t(j) waits for its P·V MMAs; at
  // D = 128 the 512 columns are full and P is written over S.
  static constexpr bool SEP_P = D <= 64;
  static constexpr int COL_P0 = SEP_P ? 256 + 2 * D : COL_S0;
  static constexpr int COL_P1 = SEP_P ? 256 + 2 * D + 64 : COL_S1;
  static_assert(!SEP_P || COL_P1 + 64 <= TMEM_COLS, "tensor-memory columns");
  static constexpr int THREADS = 384;
  // Launch: 168 registers x 384 threads.  The softmax warpgroups (0, 1)
  // rise to REGS_SOFTMAX, warpgroup 2 (producer, MMA, copier or second MMA)
  // drops to REGS_OTHER; the sum stays within 384*168, so the increase never
  // waits on registers that do not exist.
#ifndef FA_REGS_SOFTMAX
#define FA_REGS_SOFTMAX 184
#define FA_REGS_OTHER 136
#endif
  static constexpr int REGS_SOFTMAX = FA_REGS_SOFTMAX;
  static constexpr int REGS_OTHER = FA_REGS_OTHER;
  static_assert(2 * 128 * REGS_SOFTMAX + 128 * REGS_OTHER <= THREADS * 168, "register split");
};

// Kernel parameters.  The scalars every role reads to decode its work units
// come first, within the first 64 bytes, then the other scalars and pointers,
// then the three tensor maps (64-byte aligned): a CTA's first reads of its
// parameters miss the constant cache, and fewer distinct lines mean fewer
// serial misses before the first copy is issued.
struct Params {
  // -- unit decode (first line) --
  int num_units;       // BH * units_per_bh * num_splits
  int tail_start;      // units >= tail_start are single query tiles (halves of the
                       // last pair units; unsplit launches only), else == num_units
  int units_per_bh;    // ceil(ceil(Nq/128)/2)
  int num_splits;      // key ranges computed separately (1 = no split), <= nkv
  int nkv;             // ceil(Nk/128): key blocks in all
  int causal;          // exclude key j > query i
  int BH, H, Nq, Nk;
  int seg;             // > 0: rows and keys form consecutive segments of this length
                       // and a row sees only keys of its own segment (packed windows)
  int inject_stall;    // test hook: CTA 0's producer withholds its 4th K/V tile
  FastDiv div_upb;     // division by units_per_bh
  FastDiv div_splits;  // by num_splits
  FastDiv div_bh;      // by BH
  FastDiv div_h;       // by H
  unsigned long long timeout_ns;
  // -- softmax and epilogue --
  float scale_log2;    // scale * log2(e)
  int mask_kind;       // how the general softmax path reads mask values (kMask*): selects
                       // the kernel instantiation
  int full_mask_bool;  // 0: additive fp32; 1: uint8, nonzero = keep, 0 = -inf
  int mask_heads;      // 1 (broadcast over heads) or H
  int qtiles;          // ceil(Nq/128)
  int* status;         // device status word: set to FA_ERR_TIMEOUT when a wait runs out
  int* debug_record;   // debug builds: first failed device-side check (8 ints)
  int debug_plant;     // debug builds, test hook: the O-store check uses bound Nq - 1
  __nv_bfloat16* out;  // [BH][Nq][D]
  float* lse;          // [BH][Nq]
  const float* mask;   // key padding [B][Nk] or nullptr
  const void* full_mask;  // per (query, key) mask [B][mask_heads][Nq][Nk] or nullptr
  float* part_o;       // split mode: fp32 [num_splits][BH][Nq][D] partial O (else nullptr)
  float* part_lse;     // split mode: fp32 [num_splits][BH][Nq] partial LSE
  const float* q_scale;   // F8: [BH][ceil(Nq/128)] e4m3 block scale of Q
  const float* k_scale;   // F8: [BH][nkv] e4m3 block scale of the smoothed K
  const float* lse_corr;  // F8: [BH][Nq] scale * q_i . mean(K), added back to LSE
  // Window mode (win != 0; the kernel's WIN instantiation): the launch is the
  // batched problem over windows ([entries][H][entry tokens], see WindowGeom)
  // but Q, K, V are read from the original [B][H][tokens][D] tensors and O,
  // LSE written to the original [B][H][tokens] rows, each windowed row through
  // WindowGeom::source_row.
  int win;
  WindowGeom wg;
  const __nv_bfloat16* win_q;
  const __nv_bfloat16* win_k;
  const __nv_bfloat16* win_v;
  // -- TMA descriptors (each 64-byte aligned) --
  CUtensorMap tm_q;  // [BH][Nq][D] bf16 (e4m3 for the F8 kernel)
  CUtensorMap tm_k;  // [BH][Nk][D]
  CUtensorMap tm_v;  // [BH][Nk][D]
  CUtensorMap tm_mask;  // staged mask kind: [B][mask_heads][Nq][Nk] fp32
};
static_assert(sizeof(Params) <= 4096, "kernel parameter space");


// One work unit: nq query tiles (256 rows, or 128 at the Nq tail and in the
// last wave) of one (b, h) against one range of key blocks.
struct Unit {
  int bh, q0, nq, split, tile0, ntiles;
};

// Units are numbered head-major, then query pair, then key range, so CTAs
// running together share a head's K/V (and Q) in L2.  When the pair units do
// not fill the last wave of the persistent grid, the last ones are split into
// single-tile units (two per pair, numbered from tail_start) so that wave is
// shorter.
__device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
  Unit r;
  const uint32_t upb = (uint32_t)p.units_per_bh;
  // Pair index -> (head, first query row), head-major.
  auto locate = [&](uint32_t pair, int& bh, int& q0) {
    const uint32_t k = p.div_upb.div(pair);
    bh = (int)k;
    q0 = (int)(pair - k * upb) * 256;
  };
  if (u >= p.tail_start) {
    const uint32_t v = (uint32_t)(u - p.tail_start);
    const uint32_t pair = (uint32_t)p.tail_start + (v >> 1);  // unsplit launch: unit == pair index
    locate(pair, r.bh, r.q0);
    r.split = 0;
    r.q0 += (int)(v & 1) * 128;
    r.nq = 1;
  } else if (p.causal) {
    // Causal (one key range): a pair's work grows with its query position, so
    // units run heaviest first.  When a head has fewer pairs than the grid has
    // CTAs, across all heads (pair index descending, heads inner): each round
    // then holds units of equal weight, and dealt to the CTAs in snake order
    // (snake_unit) the CTAs' totals stay close.  When a head has at least a
    // round of pairs, head by head (heaviest first within each head): the
    // CTAs running together then sweep one head's keys, which stay in L2,
    // where heads inner would stream every head's K/V at once; the snake
    // order pairs each round's heavy end with the next round's light end.
    r.split = 0;
    if (p.units_per_bh >= (int)gridDim.x) {
      const uint32_t k = p.div_upb.div((uint32_t)u);
      r.bh = (int)k;
      r.q0 = (int)(upb - 1 - ((uint32_t)u - k * upb)) * 256;
    } else {
      const uint32_t k = p.div_bh.div((uint32_t)u);
      r.bh = u - (int)k * p.BH;
      r.q0 = (int)(upb - 1 - k) * 256;
    }
    r.nq = (r.q0 + 128 < p.Nq) ? 2 : 1;
  } else {
    uint32_t rest = (uint32_t)u;
    r.split = 0;
    if (p.num_splits > 1) {
      rest = p.div_splits.div((uint32_t)u);
      r.split = u - (int)rest * p.num_splits;
    }
    locate(rest, r.bh, r.q0);
    r.nq = (r.q0 + 128 < p.Nq) ? 2 : 1;
  }
  if (p.num_splits == 1) {
    r.tile0 = 0;
    r.ntiles = p.nkv;
  } else {
    // Balanced ranges: range s covers key blocks [s*nkv/S, (s+1)*nkv/S).
    r.tile0 = (int)((long long)r.split * p.nkv / p.num_splits);
    r.ntiles = (int)((long long)(r.split + 1) * p.nkv / p.num_splits) - r.tile0;
  }
  if (p.causal) {
    // Key blocks past the unit's last query row are fully masked: skip them
    // (causal launches use one key range, so at least one block remains).
    const int last_row = min(r.q0 + 128 * r.nq - 1, p.Nq - 1);
    r.ntiles = min(r.ntiles, last_row / 128 + 1 - r.tile0);
  }
  return r;
}

// The CTA's ui-th unit.  Units are dealt to the persistent CTAs round by
// round, in ascending CTA order in even rounds and descending order in odd
// ones (a snake): with units sorted heaviest first (causal launches) each
// CTA's total stays near the mean, where a plain round-robin gives CTA 0 the
// heaviest unit of every round; a round's set of units (what runs together,
// sharing L2) is unchanged.  Past INT_MAX the index saturates (>= num_units).
__device__ __forceinline__ int snake_unit(int ui) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long v = (long long)ui * G + ((ui & 1) ? G - 1 - c : c);
  return v > INT_MAX ? INT_MAX : (int)v;
}

// Host side of the unit schedule, last-wave balancing: with P pair units on
// G persistent CTAs, the final wave holds R = P mod G of them.  If R <= G/2,
// those R pairs run as 2R single-tile units instead (numbered from
// tail_start), one per CTA, which finish sooner than pairs.  Only for unsplit,
// non-causal launches whose heads have an even number of query tiles (every
// pair unit then holds two tiles; causal launches order their units heaviest
// first instead).
inline void plan_last_wave(Params& prm, int G) {
  prm.tail_start = prm.num_units;
  if (prm.num_splits == 1 && !prm.causal && ((prm.Nq + 127) / 128) % 2 == 0 &&
      prm.num_units > G && prm.num_units <= INT_MAX - G) {
    const int R = prm.num_units % G;
    if (R > 0 && 2 * R <= G) {
      prm.tail_start = prm.num_units - R;
      prm.num_units += R;
    }
  }
}

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start
// address, leading / stride byte offsets (16-byte units), version 1,
// swizzle layout in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)layout << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulate.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor for kind::f8f6f4 with e4m3 A/B (format 0), K-major,
// fp32 accumulate.
__host__ __device__ constexpr uint32_t make_idesc_f8(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t s_full[2], p_half[2], p_ready[2], o_full[2];
  uint64_t s_free[2], pv_done[2];  // separate-P schedule (D <= 64)
  uint64_t drain1;                 // the second MMA warp's drain (D <= 64)
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t m_full[kMaskFullBars], m_empty[kMaskSlots];  // staged mask pieces
  int dbg_unit[3];  // debug builds: (unit, bh, q0) the producer loaded Q for
};

// Device-side checks of a debug build (-DFA_DEBUG): every global access and
// the unit schedule are checked before use.  A failed check records the
// first violation (check id, CTA, thread, two values; a count of failures),
// sets FA_ERR_DEBUG_CHECK in the status word and the CTA's abort flag (so
// every later wait returns and the CTA drains as after a timeout), and the
// access is skipped.  Release builds compile every check to `true`.
__device__ __forceinline__ bool fa_check(const Params& p, Barriers* bars, bool cond, int id,
                                         long long a, long long b) {
#ifdef FA_DEBUG
  if (!cond) {
    atomicCAS(p.status, 0, kStatusDebugCheck);
    if (atomicCAS(&p.debug_record[0], 0, id) == 0) {
      p.debug_record[1] = (int)blockIdx.x;
      p.debug_record[2] = (int)threadIdx.x;
      p.debug_record[3] = (int)a;
      p.debug_record[4] = (int)b;
    }
    atomicAdd(&p.debug_record[7], 1);
    bars->abort_flag = 1;
  }
  return cond;
#else
  (void)p; (void)bars; (void)id; (void)a; (void)b;
  return cond || true;
#endif
}

// Check ids.
enum : int {
  kCheckUnit = 1,       // decoded unit inside the problem (head, query pair, key blocks)
  kCheckUnitSync = 2,   // the MMA warp's unit equals the one the producer loaded
  kCheckMaskRow = 3,    // mask row inside the mask array
  kCheckScale = 4,      // e4m3 block-scale index inside its array
  kCheckStore = 5,      // O / LSE / partial store inside its array
};

// A decoded unit lies inside the problem.
__device__ __forceinline__ bool unit_in_bounds(const Params& p, const Unit& un) {
  return un.bh >= 0 && un.bh < p.BH && un.q0 >= 0 && un.q0 < p.Nq && (un.q0 & 127) == 0 &&
         (un.nq == 1 || un.nq == 2) && un.q0 + 128 * (un.nq - 1) < p.Nq && un.tile0 >= 0 &&
         un.ntiles >= 1 && un.tile0 + un.ntiles <= p.nkv && un.split >= 0 &&
         un.split < p.num_splits;
}

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting
// (this wait ran out of time, or another one did).  Between polls the thread
// sleeps in try_wait (woken when the phase completes).
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, Barriers* bars,
                                             unsigned long long timeout_ns, int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
    if (bars->abort_flag) return false;
    if (ptx::global_timer_ns() - t0 > timeout_ns) {
      bars->abort_flag = 1;
      atomicCAS(status, 0, kStatusTimeout);
      return false;
    }
  }
}

// Warp-uniform version: every lane waits, then the warp agrees.  A phase
// that has already completed is taken with one test and one vote.
__device__ __forceinline__ bool bounded_wait_warp(uint32_t bar, uint32_t parity, Barriers* bars,
                                                  unsigned long long timeout_ns, int* status) {
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
  bool ok = bounded_wait(bar, parity, bars, timeout_ns, status);
  return __all_sync(0xffffffffu, ok);
}

// Which columns (position within a 32-column chunk, step 2) take their exp2 on
// the FMA pipe instead of the MUFU unit: FA_EMU_PAIRS of the 16 pairs.  Off
// by default: on GB300 every share tried (2/16 .. 8/16 pairs) was slower than
// none, the extra issue slots costing more than the MUFU time saved.
#ifndef FA_EMU_PAIRS
#define FA_EMU_PAIRS 0
#endif
__host__ __device__ constexpr bool kEmulatedExp2(int c) { return (c / 2) % 16 < FA_EMU_PAIRS; }

// 2^x for a pair of fp32 values on the FMA pipe (Cody–Waite style range
// reduction plus a polynomial): x = n + f with n = round(x) (by adding
// 1.5·2^23, whose low mantissa bits then hold n) and f in [-1/2, 1/2];
// 2^f ≈ c0 + c1 f + c2 f² + c3 f³ with coefficients from a Remez (minimax
// relative error) fit on [-1/2, 1/2] — max relative error 7.5e-5, below the
// bf16 rounding of P (2^-9); n is added into the exponent field.  x is
// clamped at -126 so the result stays a non-negative float (the true value
// there is below 2^-125 and does not matter next to the row maximum 2^0).
__device__ __forceinline__ float2 exp2_fma_pipe(float2 x) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  constexpr float c0 = 0.99992805719375610f, c1 = 0.69326096773147583f;
  constexpr float c2 = 0.24261112511157990f, c3 = 0.05517166852951050f;
  x.x = fmaxf(x.x, -126.f);
  x.y = fmaxf(x.y, -126.f);
  const float2 j = __fadd2_rn(x, make_float2(kRound, kRound));
  const float2 n = __fadd2_rn(j, make_float2(-kRound, -kRound));
  const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), x);
  float2 q = __ffma2_rn(f, make_float2(c3, c3), make_float2(c2, c2));
  q = __ffma2_rn(q, f, make_float2(c1, c1));
  q = __ffma2_rn(q, f, make_float2(c0, c0));
  const uint32_t b0 = __float_as_uint(q.x) + (__float_as_uint(j.x) << 23);
  const uint32_t b1 = __float_as_uint(q.y) + (__float_as_uint(j.y) << 23);
  return make_float2(__uint_as_float(b0), __uint_as_float(b1));
}

// Mask values of one 16-key step of the general softmax path (keys
// key0 .. key0 + 15 of the row `mrow`): 16 fp32 values, or 16 bytes packed
// four to a word in w[0..3].  Every index is clamped inside the row (values
// past Nk are never used: the key range excludes them).
constexpr int kGenStep = 16;
template <int MK>
__device__ __forceinline__ void general_load(const void* mrow, int key0, int Nk,
                                             uint32_t (&w)[kGenStep]) {
  const float* mf = static_cast<const float*>(mrow);
  const uint8_t* mb = static_cast<const uint8_t*>(mrow);
  if constexpr (MK == kMaskF32Scalar) {
#pragma unroll
    for (int i = 0; i < kGenStep; ++i) w[i] = __float_as_uint(__ldg(mf + min(key0 + i, Nk - 1)));
  } else if constexpr (MK == kMaskU8Vec) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(mb + min(key0, Nk - 16)));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (MK == kMaskU8Scalar) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t x = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) x |= (uint32_t)__ldg(mb + min(key0 + 4 * k + b, Nk - 1)) << (8 * b);
      w[k] = x;
    }
  }
}

// Pass 1 of the general softmax path for one key block: each of the row's
// scores s (tensor memory, 16 columns per step) becomes the log2-domain value
// t = s * sl2 + add * log2(e), or -inf outside the row's valid keys
// [lo, lo + span) of the block (the Nk tail, the causal diagonal, the
// segment of a packed window).  A uint8 mask value 0 excludes its key; an
// fp32 value is added.  t is written back over s; the row max of t is
// returned.  Only the first `nsteps` steps (an even number, uniform across the
// warp) are processed: the caller guarantees that no row of the warp has a
// valid key past them.  Neither loop branches per key (exclusion is a range
// compare and a select); the steps run in pairs with two buffers of mask
// values (a, b), each refilled right after its step, two steps ahead of its
// next use.  `a` and `b` hold steps 0 and 1, loaded by the caller before S
// was ready.
template <int MK>
__device__ __forceinline__ float general_pass1(uint32_t tS, const void* mrow, int kbase, int Nk,
                                               int lo, uint32_t span, float sl2, int nsteps,
                                               uint32_t (&a)[kGenStep], uint32_t (&b)[kGenStep]) {
  constexpr float kLog2e = 1.4426950408889634f;
  float mx = -INFINITY;
  // 16 scores of r (starting at column cb) with the mask values w.
  auto step = [&](int cb, uint32_t* r, const uint32_t (&w)[kGenStep]) {
    const int d = cb - lo;
#pragma unroll
    for (int i = 0; i < kGenStep; ++i) {
      float t = __uint_as_float(r[i]) * sl2;
      bool keep = (uint32_t)(d + i) < span;
      if constexpr (MK == kMaskF32Scalar) {
        t = fmaf(__uint_as_float(w[i]), kLog2e, t);
      } else if constexpr (MK == kMaskU8Vec || MK == kMaskU8Scalar) {
        keep = keep && ((w[i / 4] >> (8 * (i % 4))) & 0xffu) != 0u;
      }
      t = keep ? t : -INFINITY;
      mx = fmaxf(mx, t);
      r[i] = __float_as_uint(t);
    }
  };
  const int end = nsteps * kGenStep;
#pragma unroll 1
  for (int cb = 0; cb < end; cb += 2 * kGenStep) {
    // One tensor-memory round trip per pair of steps.  Each buffer is
    // refilled as soon as its step has used it, with the keys it serves two
    // steps later (clamped to the block: the last pair reloads its own keys,
    // which are never used).
    const int nb = kbase + min(cb + 2 * kGenStep, 128 - 2 * kGenStep);
    uint32_t r[2 * kGenStep];
    ptx::tmem_ld32x32b_x32(tS + cb, r);
    step(cb, r, a);
    general_load<MK>(mrow, nb, Nk, a);
    step(cb + kGenStep, r + kGenStep, b);
    general_load<MK>(mrow, nb + kGenStep, Nk, b);
    ptx::tmem_st32x32b_x32(tS + cb, r);
  }
  return mx;
}

// Pass 1 of the general path for a key-padding mask with Nk a multiple of 4
// (kMaskF32Vec): as general_pass1, with the block's 128 mask values already
// in registers across the warp (lane l holds keys 4l .. 4l + 3 of the block
// in kv; clamped inside the row, so lanes past Nk hold values the key range
// excludes).  Every row of the warp reads the same keys, so each 32-key step
// takes its values by shuffles from lanes cb/4 .. cb/4 + 7.
__device__ __forceinline__ float general_pass1_key4(uint32_t tS, float4 kv, int lo, uint32_t span,
                                                    float sl2, int nsteps) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float2 sl22 = make_float2(sl2, sl2), l2e2 = make_float2(kLog2e, kLog2e);
  // Every row of the warp keeps every key of the block: no key-range selects.
  const bool full = __all_sync(0xffffffffu, lo == 0 && span >= 128u);
  float mx = -INFINITY;
  const int end = nsteps * kGenStep;  // nsteps is even: 32 keys per iteration
#pragma unroll 1
  for (int cb = 0; cb < end; cb += 2 * kGenStep) {
    uint32_t r[2 * kGenStep];
    ptx::tmem_ld32x32b_x32(tS + cb, r);
    const int d = cb - lo;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int src = (cb >> 2) + q;
      const float mv[4] = {__shfl_sync(0xffffffffu, kv.x, src), __shfl_sync(0xffffffffu, kv.y, src),
                           __shfl_sync(0xffffffffu, kv.z, src), __shfl_sync(0xffffffffu, kv.w, src)};
#pragma unroll
      for (int e = 0; e < 4; e += 2) {  // f32x2 pairs
        const int i = 4 * q + e;
        float2 t = __ffma2_rn(make_float2(mv[e], mv[e + 1]), l2e2,
                              __fmul2_rn(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                         sl22));
        if (!full) {
          t.x = (uint32_t)(d + i) < span ? t.x : -INFINITY;
          t.y = (uint32_t)(d + i + 1) < span ? t.y : -INFINITY;
        }
        mx = ptx::fmax3(mx, t.x, t.y);
        r[i] = __float_as_uint(t.x);
        r[i + 1] = __float_as_uint(t.y);
      }
    }
    ptx::tmem_st32x32b_x32(tS + cb, r);
  }
  return mx;
}

// Pass 1 of the general path for a staged fp32 mask (kMaskF32Staged): as
// general_pass1, with the row's mask values read from the shared-memory
// pieces the mask producer filled.  A piece is 16 KB: 128 rows x 32 fp32
// keys (128 bytes), 128-byte swizzle: 16-byte chunk c of row r sits at chunk
// c ^ (r mod 8), so a warp's 32 rows read distinct bank groups.  Pieces
// piece0 .. piece0 + 3 of the producer's sequence hold this block's keys for
// this tile; piece i is in slot i mod kMaskSlots, signalled on full barrier
// i mod kMaskFullBars.  Each is waited for, read (only its steps below
// `nsteps`), and released by every warp of the warpgroup (one arrive per
// warp).  Returns the row max; `ok` false if a wait ran out (the CTA is
// aborting).
__device__ __forceinline__ float general_pass1_staged(uint32_t tS, const uint8_t* sMask,
                                                      Barriers* bars, const Params& p, int row,
                                                      int lo, uint32_t span, float sl2, int nsteps,
                                                      uint32_t piece0, bool& ok) {
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr int PK = 32;                    // keys per piece
  constexpr int NP = 128 / PK;              // pieces per block
  constexpr int PB = 128 * 128;             // bytes per piece
  const uint32_t lane = threadIdx.x & 31;
  const int rsw = row & 7;
  const float2 sl22 = make_float2(sl2, sl2), l2e2 = make_float2(kLog2e, kLog2e);
  // Every row of the warp keeps every key of the block (no Nk tail, causal
  // diagonal or segment boundary in it): no key-range selects.
  const bool full = __all_sync(0xffffffffu, lo == 0 && span >= 128u);
  float mx = -INFINITY;
#pragma unroll 1
  for (int pc = 0; pc < NP; ++pc) {
    const uint32_t idx = piece0 + (uint32_t)pc;
    if (!bounded_wait_warp(ptx::smem_u32(&bars->m_full[idx % kMaskFullBars]),
                           (idx / kMaskFullBars) & 1u, bars, p.timeout_ns, p.status)) {
      ok = false;
      return mx;
    }
    const uint8_t* rowp = sMask + (idx % kMaskSlots) * PB + row * 128;
    const int cb = pc * PK;  // the piece's 32 keys in one tensor-memory round trip
    if (cb < nsteps * kGenStep) {
      uint32_t r[PK];
      ptx::tmem_ld32x32b_x32(tS + cb, r);
      const int d = cb - lo;
      // Scores and mask values in f32x2 pairs; the key-range selects only
      // where some row of the warp does not keep the whole block.
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {  // 16-byte chunks of the row's 128 bytes
        const uint4 v = *reinterpret_cast<const uint4*>(rowp + ((ch ^ rsw) << 4));
        const float w[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                            __uint_as_float(v.w)};
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int i = 4 * ch + e;
          float2 t = __ffma2_rn(make_float2(w[e], w[e + 1]), l2e2,
                                __fmul2_rn(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                           sl22));
          if (!full) {
            t.x = (uint32_t)(d + i) < span ? t.x : -INFINITY;
            t.y = (uint32_t)(d + i + 1) < span ? t.y : -INFINITY;
          }
          mx = ptx::fmax3(mx, t.x, t.y);
          r[i] = __float_as_uint(t.x);
          r[i + 1] = __float_as_uint(t.y);
        }
      }
      ptx::tmem_st32x32b_x32(tS + cb, r);
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->m_empty[idx % kMaskSlots]));
  }
  return mx;
}

// Window mode: one 128-row bf16 tile, windowed rows row0 .. row0 + 127 (rows
// from nvalid on repeat row nvalid - 1, whose results are discarded), copied
// by the whole warp from the original tensor `src` with cp.async (16 bytes
// per lane per instruction, consecutive lanes on consecutive pieces of a
// row) into the layout a TMA tile load writes: 128-row chunk blocks of SW-byte
// rows, 16-byte piece c of row r at piece c ^ (r mod 8) (128-byte swizzle) or
// c ^ ((r / 2) mod 4) (64-byte swizzle).  Each lane maps four rows (lane,
// lane + 32, ...) and the others take them by shuffle.
template <int D>
__device__ __forceinline__ void window_tile(const WindowGeom& g, const __nv_bfloat16* src,
                                            uint32_t row0, int nvalid, uint32_t dst, uint32_t lane) {
  constexpr int SW = (D >= 64) ? 128 : 64;
  constexpr int CPR = D / 8;      // 16-byte pieces per row
  constexpr int CPB = SW / 16;    // pieces per swizzled row of a chunk block
  constexpr int RPI = 32 / CPR;   // rows per instruction
  uint32_t srow[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = k * 32 + (int)lane;
    srow[k] = (uint32_t)g.source_row(row0 + (uint32_t)(r < nvalid ? r : nvalid - 1));
  }
#pragma unroll
  for (int k = 0; k < 128 / RPI; ++k) {
    const int r = k * RPI + (int)lane / CPR;
    const int c = (int)lane % CPR;
    const uint32_t sr = __shfl_sync(0xffffffffu, srow[(k * RPI) / 32], r % 32);
    const __nv_bfloat16* gp = src + (size_t)sr * D + c * 8;
    const int swz = SW == 128 ? (r & 7) : ((r >> 1) & 3);
    const uint32_t so = dst + (uint32_t)((c / CPB) * (128 * SW) + r * SW + (((c % CPB) ^ swz) << 4));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(so), "l"(gp) : "memory");
  }
}

// MK: how the general softmax path reads mask values (kMask*).  Each kind is
// its own instantiation, so a launch carries only the mask code it runs (the
// kernel's speed is sensitive to its instruction footprint).  WIN: window mode
// (rows gathered and scattered through the window map; Params::win).
template <int D, bool F8, int MK, bool WIN>
__global__ void __launch_bounds__(Cfg<D, F8, MK>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ Params p) {
  using C = Cfg<D, F8, MK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // 2 tiles
  uint8_t* sMask = smem + C::SMEM_Q;           // staged mask kind: MASK_SLOTS pieces
  uint8_t* sRing = sMask + C::SMEM_MASK;       // STAGES tiles
  uint8_t* sEpi = sRing + C::SMEM_RING;       // D <= 64: output staging, 8 warps
  Barriers* bars = reinterpret_cast<Barriers*>(sEpi + C::SMEM_EPI);

  const int warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->q_empty), C::SEP_P ? 2 : 1);  // one per MMA warp
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[t]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->p_half[t]), 128);
      ptx::mbar_init(ptx::smem_u32(&bars->p_ready[t]), 128);
      ptx::mbar_init(ptx::smem_u32(&bars->o_full[t]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->s_free[t]), 4);  // one arrive per softmax warp
      ptx::mbar_init(ptx::smem_u32(&bars->pv_done[t]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain1), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->kv_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->kv_empty[s]), C::SEP_P ? 2 : 1);
    }
    if constexpr (C::STAGED_MASK) {
      for (int s = 0; s < C::MASK_FULL_BARS; ++s) ptx::mbar_init(ptx::smem_u32(&bars->m_full[s]), 1);
      for (int s = 0; s < C::MASK_SLOTS; ++s)
        ptx::mbar_init(ptx::smem_u32(&bars->m_empty[s]), 4);  // one arrive per consuming warp
    }
    bars->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  // Every role ends here (its own inlined copy, so code running under
  // different register limits never merges): all warps meet, then the TMEM
  // owner frees the columns.
  auto finish = [&]() {
    ptx::named_barrier_sync(1, C::THREADS);
    if (warp == 9) {
      ptx::tc_fence_after_sync();
      ptx::tmem_dealloc(tmem, C::TMEM_COLS);
    }
  };

  if (warp >= 8) {
  // Warpgroup 2 gives registers to the softmax warpgroups (same PC for its
  // four warps; code under different register limits never shares a path).
  ptx::setmaxnreg_dec<C::REGS_OTHER>();
  if (warp == 8) {
    // ------------------------------------------------------------ producer --
    if constexpr (WIN) {
      // Window mode: the whole warp gathers tiles with cp.async.  A tile's
      // copies form one group; once at most kInFlight later groups are
      // pending it has landed, and each lane fences its writes for the tensor
      // cores (async proxy) before lane 0 arrives on the tile's barrier.
      // Before waiting for the Q buffer every group is flushed (the MMA needs
      // all of the last unit's K tiles to release Q).
      constexpr int kInFlight = 2;
      uint32_t pd0 = 0, pd1 = 0, pd2 = 0;  // barriers of pending groups, oldest first
      int np = 0;
      auto arrive_oldest = [&]() {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(pd0);
        pd0 = pd1;
        pd1 = pd2;
        --np;
      };
      auto commit = [&](uint32_t bar) {
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (np == 0) pd0 = bar; else if (np == 1) pd1 = bar; else pd2 = bar;
        ++np;
        if (np > kInFlight) {
          asm volatile("cp.async.wait_group %0;" ::"n"(kInFlight) : "memory");
          arrive_oldest();
        }
      };
      auto flush = [&]() {
        asm volatile("cp.async.wait_all;" ::: "memory");
        while (np > 0) arrive_oldest();
      };
      const uint32_t sq = ptx::smem_u32(sQ), sring = ptx::smem_u32(sRing);
      uint32_t it = 0, uc = 0;
      bool ok = true;
      for (int ui = 0, u = snake_unit(0); u < p.num_units && ok; u = snake_unit(++ui), ++uc) {
        const Unit un = decode_unit(p, u);
        const int bh = un.bh, q0 = un.q0;
        flush();
        ok = bounded_wait_warp(ptx::smem_u32(&bars->q_empty), (uc & 1) ^ 1, bars, p.timeout_ns, p.status);
        if (!ok) break;
        if (!fa_check(p, bars, unit_in_bounds(p, un), kCheckUnit, u, un.bh)) {
          ok = false;
          break;
        }
#ifdef FA_DEBUG
        if (lane == 0) {
          bars->dbg_unit[0] = u;
          bars->dbg_unit[1] = bh;
          bars->dbg_unit[2] = q0;
        }
#endif
        for (int t = 0; t < un.nq; ++t)
          window_tile<D>(p.wg, p.win_q, (uint32_t)(bh * p.Nq + q0 + t * 128), p.Nq - (q0 + t * 128),
                         sq + t * C::QK_TILE_BYTES, lane);
        commit(ptx::smem_u32(&bars->q_full));
        for (int j = 0; j < un.ntiles && ok; ++j) {
          const int kb = (un.tile0 + j) * 128;
          for (int kv = 0; kv < 2; ++kv, ++it) {
            const uint32_t s = it % C::STAGES;
            const uint32_t ph = (it / C::STAGES) & 1;
            ok = bounded_wait_warp(ptx::smem_u32(&bars->kv_empty[s]), ph ^ 1, bars, p.timeout_ns, p.status);
            if (!ok) break;
            window_tile<D>(p.wg, kv ? p.win_v : p.win_k, (uint32_t)(bh * p.Nk + kb), p.Nk - kb,
                           sring + s * C::TILE_BYTES, lane);
            commit(ptx::smem_u32(&bars->kv_full[s]));
          }
        }
      }
      if (ok)
        flush();
      else
        asm volatile("cp.async.wait_all;" ::: "memory");  // nothing lands after the CTA ends
    } else if (lane == 0) {
      ptx::tma_prefetch_desc(&p.tm_q);
      ptx::tma_prefetch_desc(&p.tm_k);
      ptx::tma_prefetch_desc(&p.tm_v);
      uint32_t it = 0, uc = 0;        // K/V tiles handled so far, units started
      uint32_t skipped = 0xffffffffu;  // the tile the stall hook withheld, if any
      uint32_t q_issued = 0;
      bool ok = true;
      for (int ui = 0, u = snake_unit(0); u < p.num_units && ok; u = snake_unit(++ui), ++uc) {
        const Unit un = decode_unit(p, u);
        const int bh = un.bh, q0 = un.q0;
        const int ntiles = un.nq;
        ok = bounded_wait(ptx::smem_u32(&bars->q_empty), (uc & 1) ^ 1, bars, p.timeout_ns, p.status);
        if (!ok) break;
        if (!fa_check(p, bars, unit_in_bounds(p, un), kCheckUnit, u, un.bh)) {
          ok = false;  // drain this thread's copies in flight, as after a timeout
          break;
        }
#ifdef FA_DEBUG
        bars->dbg_unit[0] = u;
        bars->dbg_unit[1] = bh;
        bars->dbg_unit[2] = q0;
#endif
        const uint32_t qbar = ptx::smem_u32(&bars->q_full);
        ptx::mbar_arrive_expect_tx(qbar, ntiles * C::QK_TILE_BYTES);
        for (int t = 0; t < ntiles; ++t)
          for (int c = 0; c < C::QK_NCHUNK; ++c)
            ptx::tma_load_3d(ptx::smem_u32(sQ + t * C::QK_TILE_BYTES + c * C::QK_CHUNK_BYTES),
                             &p.tm_q, qbar, c * C::QK_CHUNK_ELEMS, q0 + t * 128, bh);
        ++q_issued;
        for (int j = 0; j < un.ntiles && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++it) {
            const uint32_t s = it % C::STAGES;
            const uint32_t ph = (it / C::STAGES) & 1;
            ok = bounded_wait(ptx::smem_u32(&bars->kv_empty[s]), ph ^ 1, bars, p.timeout_ns, p.status);
            if (!ok) break;
            const uint32_t fb = ptx::smem_u32(&bars->kv_full[s]);
            if (p.inject_stall && blockIdx.x == 0 && it == 3) {  // nothing arrives: consumers time out
              skipped = it;
              continue;
            }
            if (kv == 0) {
              ptx::mbar_arrive_expect_tx(fb, C::QK_TILE_BYTES);
              for (int c = 0; c < C::QK_NCHUNK; ++c)
                ptx::tma_load_3d(ptx::smem_u32(sRing + s * C::TILE_BYTES + c * C::QK_CHUNK_BYTES),
                                 &p.tm_k, fb, c * C::QK_CHUNK_ELEMS, (un.tile0 + j) * 128, bh);
            } else {
              ptx::mbar_arrive_expect_tx(fb, C::TILE_BYTES);
              for (int c = 0; c < C::NCHUNK; ++c)
                ptx::tma_load_3d(ptx::smem_u32(sRing + s * C::TILE_BYTES + c * C::CHUNK_BYTES),
                                 &p.tm_v, fb, c * C::CHUNK_ELEMS, (un.tile0 + j) * 128, bh);
            }
          }
        }
      }
      if (!ok) {
        // Drain: wait (bounded) until every copy this thread issued has landed.
        // Stage s received the tiles k < it with k mod STAGES == s (less the
        // withheld one); its barrier's last phase is that count minus one.
        const unsigned long long t_drain = p.timeout_ns;
        for (int s = 0; s < C::STAGES; ++s) {
          uint32_t n = it > (uint32_t)s ? (it - 1 - s) / C::STAGES + 1 : 0;
          if (skipped < it && skipped % C::STAGES == (uint32_t)s) --n;
          if (n == 0) continue;
          const uint32_t bar = ptx::smem_u32(&bars->kv_full[s]);
          uint64_t t0 = ptx::global_timer_ns();
          while (!ptx::mbar_try_wait(bar, (n - 1) & 1) && ptx::global_timer_ns() - t0 < t_drain) {
          }
        }
        if (q_issued) {
          const uint32_t bar = ptx::smem_u32(&bars->q_full);
          uint64_t t0 = ptx::global_timer_ns();
          while (!ptx::mbar_try_wait(bar, (q_issued - 1) & 1) &&
                 ptx::global_timer_ns() - t0 < t_drain) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 9 || (C::SEP_P && warp == 11)) {
    // ----------------------------------------------------------------- MMA --
    // The whole warp runs the loop (operands warp-uniform); one elected lane
    // issues each MMA batch and commit.  With separate P columns (D <= 64)
    // two warps share the work: warp 9 issues tile 0's MMAs, warp 11 tile
    // 1's (a single issuing warp spends more time per key block on its
    // barrier waits, issues and commits than the softmax does at D <= 64).
    {
      constexpr uint32_t IDESC_QK = F8 ? make_idesc_f8(128, 128) : make_idesc(128, 128, false);
      constexpr uint32_t IDESC_PV = make_idesc(128, D, true);
      const uint32_t sq = ptx::smem_u32(sQ);
      const uint32_t sring = ptx::smem_u32(sRing);
      uint32_t uc = 0, pc0 = 0, pc1 = 0;
      uint32_t stage = 0, phase = 0;  // ring position as running counters (no division)
      bool ok = true;

      // Shared-memory descriptors are built once; per k-step only the start
      // address (low 14 bits, in 16-byte units) moves, which never carries
      // out of its field because shared memory is below 256 KB.
      constexpr uint32_t kTile16 = C::TILE_BYTES >> 4;       // ring stage stride
      constexpr uint32_t kQTile16 = C::QK_TILE_BYTES >> 4;   // Q tile stride
      const uint64_t dq0 = smem_desc(sq, 16, C::QK_SBO, C::QK_LAYOUT);
      const uint64_t dk0 = smem_desc(sring, 16, C::QK_SBO, C::QK_LAYOUT);
      const uint64_t dv0 = smem_desc(sring, C::CHUNK_BYTES, C::SBO, C::LAYOUT);

      const uint32_t dq_lo = (uint32_t)dq0, dq_hi = (uint32_t)(dq0 >> 32);
      const uint32_t dk_lo = (uint32_t)dk0, dk_hi = (uint32_t)(dk0 >> 32);
      const uint32_t dv_lo = (uint32_t)dv0, dv_hi = (uint32_t)(dv0 >> 32);

      // S_t = Q_t K^T : A = Q tile (K-major), B = K tile (K-major), K-dim = D;
      // one asm block per tile (the first MMA overwrites S).
      auto issue_s = [&](int t, uint32_t stg) {
        const uint32_t a = dq_lo + t * kQTile16;
        const uint32_t b = dk_lo + stg * kTile16;
        const uint32_t d = tmem + (t ? C::COL_S1 : C::COL_S0);
        if constexpr (F8) {
          if constexpr (C::S_MMAS == 4)
            ptx::mma_ss_f8_x4_el<C::s_off(1), C::s_off(2), C::s_off(3)>(d, a, dq_hi, b, dk_hi, IDESC_QK, 0);
          else if constexpr (C::S_MMAS == 2)
            ptx::mma_ss_f8_x2_el<C::s_off(1)>(d, a, dq_hi, b, dk_hi, IDESC_QK, 0);
          else
            ptx::mma_ss_f8_x1_el(d, a, dq_hi, b, dk_hi, IDESC_QK, 0);
        } else {
          if constexpr (C::S_MMAS == 8)
            ptx::mma_ss_x8_el<C::s_off(1), C::s_off(2), C::s_off(3), C::s_off(4), C::s_off(5),
                           C::s_off(6), C::s_off(7)>(d, a, dq_hi, b, dk_hi, IDESC_QK, 0);
          else if constexpr (C::S_MMAS == 4)
            ptx::mma_ss_x4_el<C::s_off(1), C::s_off(2), C::s_off(3)>(d, a, dq_hi, b, dk_hi, IDESC_QK, 0);
          else
            ptx::mma_ss_x2_el<C::s_off(1)>(d, a, dq_hi, b, dk_hi, IDESC_QK, 0);
        }
      };
      // O_t += P_t V : A = P (tensor memory: over the S_t block at D = 128,
      // its own columns at D <= 64), B = V tile (MN-major: the head dim is
      // contiguous), K-dim = 128 keys in 8 MMAs; at D = 128 issued as two
      // batches of 64 keys (the softmax releases P in halves), at D <= 64 as
      // one.  A half of P is 32 tensor-memory columns (bf16 pairs); 64 keys of
      // V are 64 rows of the V tile.
      constexpr uint32_t kVStep16 = (16 * C::SW) >> 4;
      auto issue_pv_half = [&](int t, uint32_t stg, int half, bool first) {
        const uint32_t b = dv_lo + stg * kTile16 + half * 4 * kVStep16;
        const uint32_t a_tmem = tmem + (t ? C::COL_P1 : C::COL_P0) + half * 32;
        const uint32_t d = tmem + (t ? C::COL_O1 : C::COL_O0);
        ptx::mma_ts_x4_el<kVStep16>(d, a_tmem, b, dv_hi, IDESC_PV, first ? 0u : 1u);
      };
      // Waits for each half of P_t, then issues its MMAs.  With separate P
      // columns (not on the S critical path) P is released once and its 8
      // MMAs go out together.
      auto issue_pv = [&](int t, uint32_t stg, bool first, uint32_t parity) -> bool {
        if constexpr (C::SEP_P) {
          if (!bounded_wait_warp(ptx::smem_u32(&bars->p_ready[t]), parity, bars, p.timeout_ns, p.status))
            return false;
          ptx::tc_fence_after_sync();
          ptx::mma_ts_x8_el<kVStep16>(tmem + (t ? C::COL_O1 : C::COL_O0), tmem + (t ? C::COL_P1 : C::COL_P0),
                                      dv_lo + stg * kTile16, dv_hi, IDESC_PV, first ? 0u : 1u);
          return true;
        }
        if (!bounded_wait_warp(ptx::smem_u32(&bars->p_half[t]), parity, bars, p.timeout_ns, p.status))
          return false;
        ptx::tc_fence_after_sync();
        issue_pv_half(t, stg, 0, first);
        if (!bounded_wait_warp(ptx::smem_u32(&bars->p_ready[t]), parity, bars, p.timeout_ns, p.status))
          return false;
        ptx::tc_fence_after_sync();
        issue_pv_half(t, stg, 1, false);
        return true;
      };
      // Wait until the ring's current stage is full; returns that stage.
      auto take_stage = [&](uint32_t& stg) -> bool {
        stg = stage;
        const bool r = bounded_wait_warp(ptx::smem_u32(&bars->kv_full[stage]), phase, bars, p.timeout_ns, p.status);
        if (++stage == (uint32_t)C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        ptx::tc_fence_after_sync();
        return r;
      };

      if constexpr (C::SEP_P) {
        // Separate-P schedule, one warp per tile (mt).  Per key block j:
        // S_mt(j+1) as soon as the softmax warpgroup has read its S(j) into
        // registers (s_free), so it is computed a block ahead; then
        // P_mt(j) V once the softmax releases P.  Each P V is committed to
        // pv_done[mt], which the softmax waits for before it writes P again
        // (and before its epilogue reads O).  s_free phases: one per S tile
        // the softmax has read; S tile number n (n >= 1) waits for phase n-1.
        // K/V stages and the Q buffer are released by one arrival from each
        // MMA warp; in units without a second tile warp 11 arrives without
        // MMAs (after taking the stage, so it never runs a phase ahead).
        const int mt = warp == 9 ? 0 : 1;
        uint32_t ns = 0, pcm = 0;
        auto release_stage = [&](uint32_t stg, bool mine) {
          if (mine)
            ptx::mma_commit_el(ptx::smem_u32(&bars->kv_empty[stg]));
          else if (lane == 0)
            ptx::mbar_arrive(ptx::smem_u32(&bars->kv_empty[stg]));
        };
        auto release_q = [&](bool mine) {
          if (mine)
            ptx::mma_commit_el(ptx::smem_u32(&bars->q_empty));
          else if (lane == 0)
            ptx::mbar_arrive(ptx::smem_u32(&bars->q_empty));
        };
        // S_mt for the key block in stage sK, after the softmax has read the
        // previous S_mt.
        auto next_s = [&](uint32_t sK) -> bool {
          if (ns > 0) {
            if (!bounded_wait_warp(ptx::smem_u32(&bars->s_free[mt]), (ns - 1) & 1, bars,
                                   p.timeout_ns, p.status))
              return false;
            ptx::tc_fence_after_sync();
          }
          ++ns;
          issue_s(mt, sK);
          ptx::mma_commit_el(ptx::smem_u32(&bars->s_full[mt]));
          return true;
        };
        for (int ui = 0, u = snake_unit(0); u < p.num_units && ok; u = snake_unit(++ui), ++uc) {
          const Unit un = decode_unit(p, u);
          const bool mine = mt == 0 || un.nq == 2;
          const int nkv = un.ntiles;
          ok = bounded_wait_warp(ptx::smem_u32(&bars->q_full), uc & 1, bars, p.timeout_ns, p.status);
          if (!ok) break;
#ifdef FA_DEBUG
          if (mt == 0) {
            ok = fa_check(p, bars, unit_in_bounds(p, un) && bars->dbg_unit[0] == u &&
                                       bars->dbg_unit[1] == un.bh && bars->dbg_unit[2] == un.q0,
                          kCheckUnitSync, u, bars->dbg_unit[0]);
            if (!__all_sync(0xffffffffu, ok)) break;
          }
#endif
          ptx::tc_fence_after_sync();
          uint32_t sK = 0, sV = 0;
          ok = take_stage(sK) && (!mine || next_s(sK));
          if (!ok) break;
          release_stage(sK, mine);
          if (nkv == 1) release_q(mine);
          for (int j = 0; j < nkv && ok; ++j) {
            const bool has_next = j + 1 < nkv;
            ok = take_stage(sV) && (!has_next || take_stage(sK));
            if (!ok) break;
            if (has_next) {
              if (mine) {
                ok = next_s(sK);
                if (!ok) break;
              }
              release_stage(sK, mine);
              if (j + 2 == nkv) release_q(mine);
            }
            if (mine) {
              ok = issue_pv(mt, sV, j == 0, pcm & 1);
              if (!ok) break;
              ++pcm;
              ptx::mma_commit_el(ptx::smem_u32(&bars->pv_done[mt]));
            }
            release_stage(sV, mine);
          }
        }
      } else {
        for (int ui = 0, u = snake_unit(0); u < p.num_units && ok; u = snake_unit(++ui), ++uc) {
          const Unit un = decode_unit(p, u);
          const bool has1 = un.nq == 2;
          const int nkv = un.ntiles;
          ok = bounded_wait_warp(ptx::smem_u32(&bars->q_full), uc & 1, bars, p.timeout_ns, p.status);
          if (!ok) break;
  #ifdef FA_DEBUG
          ok = fa_check(p, bars, unit_in_bounds(p, un) && bars->dbg_unit[0] == u &&
                                     bars->dbg_unit[1] == un.bh && bars->dbg_unit[2] == un.q0,
                        kCheckUnitSync, u, bars->dbg_unit[0]);
          if (!__all_sync(0xffffffffu, ok)) break;
  #endif
          ptx::tc_fence_after_sync();
          // Prologue: S for key block 0.
          uint32_t sK = 0, sV = 0;
          ok = take_stage(sK);
          if (!ok) break;
          issue_s(0, sK);
          ptx::mma_commit_el(ptx::smem_u32(&bars->s_full[0]));
          if (has1) {
            issue_s(1, sK);
            ptx::mma_commit_el(ptx::smem_u32(&bars->s_full[1]));
          }
          ptx::mma_commit_el(ptx::smem_u32(&bars->kv_empty[sK]));
          if (nkv == 1) ptx::mma_commit_el(ptx::smem_u32(&bars->q_empty));

          for (int j = 0; j < nkv && ok; ++j) {
            ok = take_stage(sV);
            if (!ok) break;
            const bool has_next = j + 1 < nkv;
            // O0 += P0 V_j
            ok = issue_pv(0, sV, j == 0, pc0 & 1);
            if (!ok) break;
            ++pc0;
            if (!has_next) ptx::mma_commit_el(ptx::smem_u32(&bars->o_full[0]));
            // S0 for key block j+1 as soon as P0 has been consumed.
            if (has_next) {
              ok = take_stage(sK);
              if (!ok) break;
              issue_s(0, sK);
              ptx::mma_commit_el(ptx::smem_u32(&bars->s_full[0]));
            }
            if (has1) {
              ok = issue_pv(1, sV, j == 0, pc1 & 1);
              if (!ok) break;
              ++pc1;
              if (!has_next) ptx::mma_commit_el(ptx::smem_u32(&bars->o_full[1]));
            }
            ptx::mma_commit_el(ptx::smem_u32(&bars->kv_empty[sV]));
            if (has_next) {
              if (has1) {
                issue_s(1, sK);
                ptx::mma_commit_el(ptx::smem_u32(&bars->s_full[1]));
              }
              ptx::mma_commit_el(ptx::smem_u32(&bars->kv_empty[sK]));
              if (j + 2 == nkv) ptx::mma_commit_el(ptx::smem_u32(&bars->q_empty));
            }
          }
        }
      }
      // Drain this thread's MMAs before tensor memory can be freed.
      {
        const uint32_t bar = ptx::smem_u32(warp == 9 ? &bars->drain : &bars->drain1);
        ptx::mma_commit_el(bar);
        uint64_t t0 = ptx::global_timer_ns();
        while (!ptx::mbar_try_wait(bar, 0) && ptx::global_timer_ns() - t0 < p.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 10) {
    // ----------------------------------------------- staged-mask producer --
    // Walks the same units and key blocks as the K/V producer and copies, for
    // every (key block, query tile), the mask pieces the softmax will read,
    // in the order it reads them (block, tile, piece), through a ring of
    // MASK_SLOTS shared-memory slots.
    if constexpr (C::STAGED_MASK) {
      if (lane == 0) {
        ptx::tma_prefetch_desc(&p.tm_mask);
        uint32_t mc = 0;  // pieces issued
        bool ok = true;
        for (int ui = 0, u = snake_unit(0); u < p.num_units && ok; u = snake_unit(++ui)) {
          const Unit un = decode_unit(p, u);
          if (!fa_check(p, bars, unit_in_bounds(p, un), kCheckUnit, u, un.bh)) {
            ok = false;
            break;
          }
          const int b = (int)p.div_h.div((uint32_t)un.bh);
          const int hm = p.mask_heads == 1 ? 0 : un.bh - b * p.H;
          for (int j = 0; j < un.ntiles && ok; ++j)
            for (int t = 0; t < un.nq && ok; ++t)
              for (int pc = 0; pc < C::MASK_PIECES; ++pc, ++mc) {
                const uint32_t slot = mc % C::MASK_SLOTS, ph = (mc / C::MASK_SLOTS) & 1u;
                ok = bounded_wait(ptx::smem_u32(&bars->m_empty[slot]), ph ^ 1u, bars, p.timeout_ns,
                                  p.status);
                if (!ok) break;
                const uint32_t fb = ptx::smem_u32(&bars->m_full[mc % C::MASK_FULL_BARS]);
                ptx::mbar_arrive_expect_tx(fb, C::MASK_PIECE_BYTES);
                ptx::tma_load_4d(ptx::smem_u32(sMask + slot * C::MASK_PIECE_BYTES), &p.tm_mask, fb,
                                 (un.tile0 + j) * 128 + pc * C::MASK_PIECE_KEYS, un.q0 + t * 128, hm,
                                 b);
              }
        }
        {
          // Wait (bounded) until every piece this thread issued has landed:
          // after an abort the softmax no longer waits for them, and the CTA
          // must not exit with copies into its shared memory in flight.
          for (uint32_t fbi = 0; fbi < (uint32_t)C::MASK_FULL_BARS; ++fbi) {
            const uint32_t n = mc > fbi ? (mc - 1 - fbi) / C::MASK_FULL_BARS + 1 : 0;
            if (n == 0) continue;
            const uint32_t bar = ptx::smem_u32(&bars->m_full[fbi]);
            uint64_t t0 = ptx::global_timer_ns();
            while (!ptx::mbar_try_wait(bar, (n - 1) & 1) &&
                   ptx::global_timer_ns() - t0 < p.timeout_ns) {
            }
          }
        }
      }
    }
    __syncwarp();
  }
  finish();  // warps 8-11
  return;
  }

  ptx::setmaxnreg_inc<C::REGS_SOFTMAX>();
  {
    // ------------------------------------------------------------- softmax --
    const int t = warp / 4;                       // query tile of this warpgroup
    const int row = (warp % 4) * 32 + lane;       // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (t ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_base + (t ? C::COL_O1 : C::COL_O0);
    const uint32_t tP = tmem + lane_base + (t ? C::COL_P1 : C::COL_P0);
    const uint32_t bar_sf = ptx::smem_u32(&bars->s_free[t]);
    const uint32_t bar_pv = ptx::smem_u32(&bars->pv_done[t]);
    const uint32_t bar_s = ptx::smem_u32(&bars->s_full[t]);
    const uint32_t bar_ph = ptx::smem_u32(&bars->p_half[t]);
    const uint32_t bar_p = ptx::smem_u32(&bars->p_ready[t]);
    const uint32_t bar_o = ptx::smem_u32(&bars->o_full[t]);
    const float scale_log2 = p.scale_log2;
    constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8
    uint32_t sc = 0, oc = 0, pvc = 0;
    // Separate-P schedule (D <= 64): S_t has been read (the MMA may write the
    // next S_t), and wait until the last P_t V has consumed P_t (before P_t is
    // written again, O_t rescaled or read by the epilogue).
    auto free_s = [&]() {
      if constexpr (C::SEP_P) {
        ptx::tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_sf);
      }
    };
    auto wait_pv = [&]() -> bool {
      if constexpr (C::SEP_P) {
        if (!bounded_wait_warp(bar_pv, pvc & 1, bars, p.timeout_ns, p.status)) return false;
        ++pvc;
        ptx::tc_fence_after_sync();
      }
      return true;
    };
    uint32_t mpiece = 0;  // staged masks: pieces of the units before this one
    bool ok = true;

    for (int ui = 0, u = snake_unit(0); u < p.num_units && ok; u = snake_unit(++ui)) {
      const Unit un = decode_unit(p, u);
      const int bh = un.bh, q0 = un.q0;
      const uint32_t unit_piece0 = mpiece;
      mpiece += (uint32_t)(un.ntiles * un.nq * C::MASK_PIECES);
      if (t == 1 && un.nq < 2) continue;
      ok = __all_sync(0xffffffffu, fa_check(p, bars, unit_in_bounds(p, un), kCheckUnit, u, bh));
      if (!ok) break;
      const int qrow = q0 + t * 128 + row;
      const int b_idx = (int)p.div_h.div((uint32_t)bh);  // batch entry of this head
      const float* mask_b = p.mask ? p.mask + (size_t)b_idx * p.Nk : nullptr;
      const bool any_full_mask = p.full_mask != nullptr;  // warp-uniform
      const int tile_row0 = q0 + t * 128;                 // first query row of this tile
      // The mask row this thread reads in the general path: the batch entry's
      // key-padding row, or its own query row of a per-(query, key) mask (rows
      // past Nq read row Nq - 1; their results are never stored).
      const void* mrow = mask_b;
      if (any_full_mask) {
        const size_t fm_row =
            ((size_t)b_idx * p.mask_heads + (p.mask_heads == 1 ? 0 : bh - b_idx * p.H)) * p.Nq +
            (size_t)min(qrow, p.Nq - 1);
        mrow = static_cast<const uint8_t*>(p.full_mask) +
               fm_row * p.Nk * (p.full_mask_bool ? 1 : sizeof(float));
        if (!fa_check(p, bars, fm_row < (size_t)(p.BH / p.H) * p.mask_heads * p.Nq, kCheckMaskRow,
                      (long long)fm_row, bh))
          mrow = p.full_mask;  // the first row: a valid address (results are discarded)
      }
      if (mask_b != nullptr &&
          !fa_check(p, bars, b_idx >= 0 && b_idx < p.BH / p.H, kCheckMaskRow, b_idx, bh))
        mask_b = p.mask;
      // Key-padding values (four keys per lane) of the unit's first key
      // block, loaded now so that their latency overlaps the unit's set-up;
      // each later block's are loaded one block ahead.
      auto load_kv = [&](int blk) {
        return __ldg(reinterpret_cast<const float4*>(
            mask_b + min((un.tile0 + blk) * 128 + 4 * (int)lane, p.Nk - 4)));
      };
      float4 kv_next = make_float4(0.f, 0.f, 0.f, 0.f);
      if (MK == kMaskF32Vec && mask_b != nullptr) kv_next = load_kv(0);
      // Keys of this row's segment (all keys when rows are not segmented).
      const int seg_lo = p.seg > 0 ? (qrow / p.seg) * p.seg : 0;
      const int seg_hi = p.seg > 0 ? seg_lo + p.seg : INT_MAX;
      float m = -INFINITY;  // running max of t_ij (log2 domain)
      float l = 0.f;        // running denominator relative to m

      for (int j = 0; j < un.ntiles; ++j) {
        const int kbase = (un.tile0 + j) * 128;
        // log2-domain multiplier of raw S; with e4m3 Q and K it carries the
        // two block scales (positive, so its sign is the sign of `scale`).
        float sl2 = scale_log2;
        if constexpr (F8) {
          const size_t qi = (size_t)bh * p.qtiles + (tile_row0 >> 7);
          const size_t ki = (size_t)bh * p.nkv + un.tile0 + j;
          if (fa_check(p, bars, qi < (size_t)p.BH * p.qtiles && ki < (size_t)p.BH * p.nkv,
                       kCheckScale, (long long)qi, (long long)ki))
            sl2 *= __ldg(p.q_scale + qi) * __ldg(p.k_scale + ki);
        }
        // Fast path: full key block, no mask, non-negative scale — the scores
        // stay in registers and the row max is taken on raw scores, scaled
        // once.  Otherwise (general path) scores are materialised in the log2
        // domain with the mask, the Nk tail, the causal diagonal and segments.
        // Blocks that need per-key work in the softmax (apart from a
        // key-padding mask, decided below once its values have arrived).
        const bool general_fixed = any_full_mask || (kbase + 128 > p.Nk) || !(sl2 >= 0.f) ||
                                   (p.causal && kbase + 127 > tile_row0) || p.seg > 0;
        // Loads issued before S is ready, so that their latency overlaps the
        // wait: the next block's key-padding values, and the general path's
        // first two steps of mask values.
        const float4 kv4 = kv_next;  // this lane's four keys of this block
        const int k4 = kbase + 4 * (int)lane;
        if (MK == kMaskF32Vec && mask_b != nullptr && j + 1 < un.ntiles) kv_next = load_kv(j + 1);
        uint32_t mwa[kGenStep], mwb[kGenStep];
        if (MK != kMaskNone && MK != kMaskF32Vec && !C::STAGED_MASK &&
            (general_fixed || mask_b != nullptr)) {
          general_load<MK>(mrow, kbase, p.Nk, mwa);
          general_load<MK>(mrow, kbase + kGenStep, p.Nk, mwb);
        }
        ok = bounded_wait_warp(bar_s, sc & 1, bars, p.timeout_ns, p.status);
        if (!ok) break;
        ++sc;
        ptx::tc_fence_after_sync();
        // A key-padding mask is classified per block (each lane checks four
        // keys, the warp votes): all zero — the block needs no mask work; all
        // excluded (-inf or past Nk) — the block contributes nothing.
        bool blk_zero = false, blk_dead = false;
        if (MK == kMaskF32Vec && mask_b != nullptr) {
          const float e[4] = {kv4.x, kv4.y, kv4.z, kv4.w};
          bool zero = true, dead = true;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool in = k4 + i < p.Nk;
            zero = zero && in && e[i] == 0.f;
            dead = dead && (!in || e[i] == -INFINITY);
          }
          blk_zero = __all_sync(0xffffffffu, zero);
          blk_dead = __all_sync(0xffffffffu, dead);
        }
        const bool general = general_fixed || (mask_b != nullptr && !blk_zero);
        auto release = [&](int h) {
          ptx::tmem_wait_st();
          ptx::tc_fence_before_sync();
          ptx::mbar_arrive(h ? bar_p : bar_ph);
        };
        // Running-max update shared by both paths (sets alpha, m_use, rescale_o).
        float alpha = 1.f, m_use = 0.f;
        bool rescale_o = false;
        auto update_max = [&](float mx) {
          const float m_new = fmaxf(m, mx);
          // Rescale only when the max grew by more than the threshold (or on the
          // first finite max); otherwise keep the stale max, which is exact
          // because the final O / l uses the same max.
          const bool grow = (m_new - m) > kRescaleThreshold;  // -inf - -inf = NaN -> false
          alpha = 1.f;
          if (grow) {
            alpha = ptx::ex2(m - m_new);  // m = -inf -> 0
            m = m_new;
          }
          m_use = (m == -INFINITY) ? 0.f : m;
          l *= alpha;
          // At D = 128, P in two halves of 64 keys, each released as soon as
          // it is in tensor memory so the first P·V MMAs overlap the second
          // half's exp2 (with separate P columns, P is released whole).  When
          // O must be rescaled (rare: the max grew past the threshold) the
          // first half waits until all of P is stored, so that the rescale
          // runs with the scores already consumed.
          rescale_o = j > 0 && __any_sync(0xffffffffu, grow);
        };
        float2 lsum = make_float2(0.f, 0.f);
        if (!general) {
          float s[128];  // the fast path keeps the scores in registers
          float mx;
          {
            uint32_t r[128];
            ptx::tmem_ld32x32b_x128(tS, r);
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(r[c]);
          }
          free_s();
          float a0 = s[0], a1 = s[1], a2 = s[2], a3 = s[3];
#pragma unroll
          for (int c = 4; c < 128; c += 8) {
            a0 = ptx::fmax3(a0, s[c], s[c + 1]);
            a1 = ptx::fmax3(a1, s[c + 2], s[c + 3]);
            a2 = ptx::fmax3(a2, s[c + 4], s[c + 5]);
            a3 = ptx::fmax3(a3, s[c + 6], s[c + 7]);
          }
          mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * sl2;
          update_max(mx);
          if (j > 0 && !wait_pv()) {
            ok = false;
            break;
          }
          const float2 sc2 = make_float2(sl2, sl2);
          const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
          for (int cb = 0; cb < 128; cb += 32) {
            uint32_t packed[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              // x <= threshold (8) by construction of the stale max.
              const float2 x = __ffma2_rn(make_float2(s[cb + c], s[cb + c + 1]), sc2, nm2);
              float2 pr;
              if (kEmulatedExp2(c)) {
                pr = exp2_fma_pipe(x);
              } else {
                pr = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
              }
              lsum = __fadd2_rn(lsum, pr);
              packed[c / 2] = ptx::pack_bf16x2(pr.x, pr.y);
            }
            ptx::tmem_st32x32b_x16(tP + cb / 2, packed);
            if (!C::SEP_P && cb == 32 && !rescale_o) release(0);
          }
        } else {
          float mx;
          // General path: two rolled loops over the S block in tensor memory
          // (this path runs on masked, causal-diagonal, Nk-tail and
          // packed-window blocks).  Pass 1 (general_pass1) turns 16 scores at a
          // time into log2-domain values with excluded pairs at -inf, keeps
          // their max and writes them back; pass 2 (below) takes their
          // exponentials.  Neither loop branches per key: a key's exclusion
          // is a range compare and a select.
          // The row's valid keys within this block: [lo, hi).
          int hi = min(128, p.Nk - kbase);
          if (p.causal) hi = min(hi, qrow - kbase + 1);
          int lo = 0;
          if (p.seg > 0) {
            lo = max(0, seg_lo - kbase);
            hi = min(hi, seg_hi - kbase);
          }
          const uint32_t span = hi > lo ? (uint32_t)(hi - lo) : 0u;
          // Steps (pairs of 16 keys) that hold a valid key for some row of
          // this warp; later columns are excluded for all 32 rows.
          // (None when the key-padding mask excludes the whole block: P = 0
          // and m, l are unchanged.)
          const int hmax = __reduce_max_sync(0xffffffffu, span ? hi : 0);
          const int nsteps = blk_dead ? 0 : min(8, 2 * ((hmax + 31) / 32));
          if constexpr (C::STAGED_MASK) {
            bool mok = true;
            mx = general_pass1_staged(tS, sMask, bars, p, row, lo, span, sl2, nsteps,
                                      unit_piece0 + (uint32_t)(j * un.nq + t) * C::MASK_PIECES, mok);
            if (!__all_sync(0xffffffffu, mok)) {
              ok = false;
              break;
            }
          } else if constexpr (MK == kMaskF32Vec) {
            mx = general_pass1_key4(tS, kv4, lo, span, sl2, nsteps);
          } else {
            mx = general_pass1<MK>(tS, mrow, kbase, p.Nk, lo, span, sl2, nsteps, mwa, mwb);
          }
          ptx::tmem_wait_st();  // pass 2 reads these columns back
          update_max(mx);
          if (j > 0 && !wait_pv()) {
            ok = false;
            break;
          }
          // Pass 2 of the general path: exponentials of the log2-domain values
          // pass 1 left in tensor memory; P (bf16 pairs) goes to P's columns
          // (at D = 128 the first 64 columns of S, behind the columns still to
          // be read).  Columns past the steps pass 1 processed are excluded
          // for every row: P = 0 there.
          // 64 columns per tensor-memory round trip where all of them hold
          // values, else 32 (pass 1 processed a multiple of 32 columns).
          const int end = nsteps * kGenStep;
          const float2 nm2 = make_float2(-m_use, -m_use);
          auto exps = [&](const uint32_t* r, uint32_t* packed, int n) {
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              if (c >= n) break;
              const float2 x =
                  __fadd2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), nm2);
              const float p0 = ptx::ex2(x.x);
              const float p1 = ptx::ex2(x.y);
              lsum = __fadd2_rn(lsum, make_float2(p0, p1));
              packed[c / 2] = ptx::pack_bf16x2(p0, p1);
            }
          };
#pragma unroll 1
          for (int cb = 0; cb < 128; cb += 64) {
            uint32_t packed[32];
            if (cb + 64 <= end) {
              uint32_t r[64];
              ptx::tmem_ld32x32b_x64(tS + cb, r);
              exps(r, packed, 64);
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c) packed[c] = 0u;
              if (cb < end) {
                uint32_t r[32];
                ptx::tmem_ld32x32b_x32(tS + cb, r);
                exps(r, packed, 32);
              }
            }
            ptx::tmem_st32x32b_x32(tP + cb / 2, packed);
            if (!C::SEP_P && cb == 0 && !rescale_o) release(0);
          }
          free_s();
        }
        l += lsum.x + lsum.y;
        if (rescale_o) {
          // P(j-1)·V has landed: the S commit that released this iteration
          // follows it (separate P: pv_done was waited for above).
#pragma unroll
          for (int cb = 0; cb < D; cb += 32) {
            uint32_t r[32];
            ptx::tmem_ld32x32b_x32(tO + cb, r);
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            ptx::tmem_st32x32b_x32(tO + cb, r);
          }
          if constexpr (!C::SEP_P) release(0);
        }
        release(1);
      }
      if (!ok) break;

      // Epilogue: O / l -> bf16, LSE = ln2 * (m + log2 l).
      if constexpr (C::SEP_P) {
        ok = wait_pv();  // the last P V of the unit: O is complete
      } else {
        ok = bounded_wait_warp(bar_o, oc & 1, bars, p.timeout_ns, p.status);
        ++oc;
      }
      if (!ok) break;
      ptx::tc_fence_after_sync();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const bool valid_row = qrow < p.Nq;
      // Output row of query row r of this head (window mode: its grid position).
      auto out_row = [&](int r) -> size_t {
        const size_t wr = (size_t)bh * p.Nq + r;
        if constexpr (WIN) return (size_t)p.wg.source_row((uint32_t)wr);
        return wr;
      };
      constexpr float kLn2 = 0.6931471805599453f;
      float row_lse = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
      if constexpr (F8) {
        // K was smoothed by its per-channel mean: add back scale * q_i . mean(K).
        if (valid_row) row_lse += __ldg(p.lse_corr + (size_t)bh * p.Nq + qrow);
      }
      if (p.part_o == nullptr && C::EPI_SMEM) {
        // Coalesced stores through shared memory: each thread writes its
        // row's D bf16 into the warp's staging buffer (16-byte chunk c of
        // row r at chunk c ^ (r mod CH), so the 32 rows' writes and the
        // reads below each take the minimum number of wavefronts), then
        // each store instruction writes 32 / CH whole rows.
        constexpr int CH = D * 2 / 16;  // 16-byte chunks per row
        uint8_t* wbuf = sEpi + warp * C::EPI_WARP_BYTES;
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
          uint32_t r[32];
          ptx::tmem_ld32x32b_x32(tO + cb, r);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = make_uint4(
                ptx::pack_bf16x2(__uint_as_float(r[8 * q]) * inv_l, __uint_as_float(r[8 * q + 1]) * inv_l),
                ptx::pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv_l, __uint_as_float(r[8 * q + 3]) * inv_l),
                ptx::pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv_l, __uint_as_float(r[8 * q + 5]) * inv_l),
                ptx::pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv_l, __uint_as_float(r[8 * q + 7]) * inv_l));
            const int c = cb / 8 + q;
            *reinterpret_cast<uint4*>(wbuf + lane * (D * 2) + ((c ^ (lane & (CH - 1))) << 4)) = v;
          }
        }
        __syncwarp();
        const int warp_row0 = q0 + t * 128 + (warp % 4) * 32;  // query row of lane 0
#pragma unroll
        for (int it = 0; it < CH; ++it) {
          const int rr = it * (32 / CH) + (int)lane / CH;  // row within the warp's 32
          const int c = (int)lane % CH;
          const uint4 v = *reinterpret_cast<const uint4*>(wbuf + rr * (D * 2) + ((c ^ (rr & (CH - 1))) << 4));
          const int orow = warp_row0 + rr;
#ifdef FA_DEBUG
          const int nq_bound = p.debug_plant ? p.Nq - 1 : p.Nq;
          if (orow < p.Nq && fa_check(p, bars, orow < nq_bound && bh < p.BH, kCheckStore,
                                      (long long)bh * p.Nq + orow, c))
#else
          if (orow < p.Nq)
#endif
            *reinterpret_cast<uint4*>(p.out + out_row(orow) * D + c * 8) = v;
        }
        __syncwarp();  // the buffer is written again in the next unit
        if (valid_row && fa_check(p, bars, bh < p.BH, kCheckStore, (long long)bh * p.Nq + qrow, -1))
          p.lse[out_row(qrow)] = row_lse;
      } else if (p.part_o == nullptr) {
        // Coalesced stores: thread = row in tensor memory, so each 32-column
        // chunk (16 bf16 pairs per row) is transposed across the warp with
        // shuffles; in pass q, lanes 4i..4i+3 write row 8q + i's 64 bytes as
        // four consecutive 16-byte pieces (8 rows per store instruction).
        const int warp_row0 = q0 + t * 128 + (warp % 4) * 32;  // query row of lane 0
        const int piece = lane & 3;                             // 16-byte piece of the row
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
          uint32_t r[32];
          ptx::tmem_ld32x32b_x32(tO + cb, r);
          uint32_t packed[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            packed[c / 2] = ptx::pack_bf16x2(__uint_as_float(r[c]) * inv_l,
                                             __uint_as_float(r[c + 1]) * inv_l);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int src = 8 * q + (lane >> 2);  // lane (= row) whose piece this lane stores
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t v = 0;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t x = __shfl_sync(0xffffffffu, packed[4 * j + k], src);
                if (piece == j) v = x;
              }
              w[k] = v;
            }
            const int orow = warp_row0 + src;
#ifdef FA_DEBUG
            const int nq_bound = p.debug_plant ? p.Nq - 1 : p.Nq;
            if (orow < p.Nq && fa_check(p, bars, orow < nq_bound && bh < p.BH, kCheckStore,
                                        (long long)bh * p.Nq + orow, cb))
#else
            if (orow < p.Nq)
#endif
              *reinterpret_cast<uint4*>(p.out + out_row(orow) * D + cb + piece * 8) =
                  make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        if (valid_row && fa_check(p, bars, bh < p.BH, kCheckStore, (long long)bh * p.Nq + qrow, -1))
          p.lse[out_row(qrow)] = row_lse;
      } else {
        // Split mode: this key range's normalised O (fp32) and its LSE, merged
        // by fa_merge_kernel.
        const size_t prow = ((size_t)un.split * p.BH + bh) * p.Nq + (valid_row ? qrow : 0);
        float* orow = p.part_o + prow * D;
        const bool prow_ok = fa_check(p, bars, prow < (size_t)p.num_splits * p.BH * p.Nq,
                                      kCheckStore, (long long)prow, -2);
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
          uint32_t r[32];
          ptx::tmem_ld32x32b_x32(tO + cb, r);
          if (valid_row && prow_ok) {
            float4* dst = reinterpret_cast<float4*>(orow + cb);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(r[4 * v4]) * inv_l,
                                    __uint_as_float(r[4 * v4 + 1]) * inv_l,
                                    __uint_as_float(r[4 * v4 + 2]) * inv_l,
                                    __uint_as_float(r[4 * v4 + 3]) * inv_l);
          }
        }
        if (valid_row && prow_ok) p.part_lse[prow] = row_lse;
      }
    }
    ptx::tc_fence_before_sync();
  }
  finish();  // softmax warps 0-7
}

// Merge of per-key-range results (the exchange step of ring attention, done
// on one GPU): for each row, LSE = log sum_s e^(LSE_s) and
// O = sum_s e^(LSE_s - LSE) O_s.  One warp per row, D/32 columns per lane;
// memory bound (reads num_splits * (D + 1) fp32 per row).
template <int D>
__global__ void __launch_bounds__(256) fa_merge_kernel(const float* __restrict__ part_o,
                                                       const float* __restrict__ part_lse,
                                                       __nv_bfloat16* __restrict__ out,
                                                       float* __restrict__ lse, int num_splits,
                                                       long long rows) {
  constexpr int PER = D / 32;
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = 0; s < num_splits; ++s) mx = fmaxf(mx, __ldg(part_lse + (long long)s * rows + row));
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < num_splits; ++s) {
      const float w = __expf(__ldg(part_lse + (long long)s * rows + row) - mx);
      wsum += w;
      const float* src = part_o + ((long long)s * rows + row) * D + lane * PER;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, __ldg(src + i), acc[i]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = out + row * D + lane * PER;
  if constexpr (PER == 1) {
    dst[0] = __float2bfloat16_rn(acc[0] * inv);
  } else {
#pragma unroll
    for (int i = 0; i < PER; i += 2)
      *reinterpret_cast<uint32_t*>(dst + i) = ptx::pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
  }
  if (lane == 0) lse[row] = (wsum > 0.f) ? mx + __logf(wsum) : -INFINITY;
}

}  // namespace fa
