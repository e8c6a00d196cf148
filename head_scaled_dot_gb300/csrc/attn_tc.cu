// attn_tc.cu - fused masked attention on tcgen05 tensor cores (bf16).
//
// A CTA takes two 128-row query tiles of one (batch item b, head i) and folds
// the allowed keys, 128 at a time, into the stable summary of every query row
// ("Stable summary of an attention key block", Definition, alphabetamath.cc):
//   m = max_j s_ij,  l = sum_j e^{s_ij - m},  z = sum_j e^{s_ij - m} v_j,
// merging each block into the running summary with
//   m' = max(m, m_blk),  l' = e^{m - m'} l + e^{m_blk - m'} l_blk,  z' likewise,
// and writes z / l once per row. The n_q x n_k score matrix only ever exists
// as one 128 x 128 block per tile, in tensor memory (TMEM).
//
// Two kernels share the units, the schedule and the TMA producers. Head sizes
// d of 72..128 run with DQK or DV = 128: Q, K and V are loaded as 64-wide
// panels and the columns past d come in as zeros (TMA fill past the tensor's
// extent), so the dot products are exact and z's extra columns stay 0.
//
// attn_tc_kernel<DQK, DV> (DV = 128, d_vh of 72..128; 384 threads):
//   warps 0, 2    TMA producers: warp 0 loads the Q tiles of each unit and the
//                 K blocks, warp 2 the V blocks, into a STAGES-deep ring (K
//                 and V freed separately); no requests ahead of the ring
//                 (L2 prefetches of the blocks past it made every workload
//                 slower)
//   warps 1, 3    MMA issuers, one per tile t: S_t = Q_t K_j^T (SMEM x SMEM
//                 -> TMEM) and z_t += P_t V_j (P from TMEM, V from SMEM); the
//                 two tiles' streams interleave on the tensor pipe, so one
//                 tile's softmax overlaps the other tile's MMAs
//   warps 4..11   softmax, tile 0 then tile 1 of every key block; a warp
//                 holds 16 rows of its 32-lane TMEM slice, lanes i and i + 16
//                 the two 64-key halves of one row (half-split TMEM loads),
//                 so the row maximum and sum take one shuffle; p is written
//                 as bf16 over the columns of S (P aliases S), and z / l at
//                 the end of the unit in the concatenated layout
//
// attn_tc_sp_kernel<DQK> (d_vh = 64; 640 threads): the same roles, but S, P
// and z of both tiles have TMEM columns of their own and each tile has its
// own eight softmax warps (warps 4..11 tile 0, 12..19 tile 1), so a tile's
// next S is computed while its softmax still works on the current one.
//
// Stale maximum: the running m of a row is only raised when a block's max
// exceeds it by more than 2^8 (then z and l are rescaled by e^{m - m'} in
// TMEM). Otherwise the block is summarised against the old m: its terms are
// e^{s - m} <= 2^8, and z / l is unchanged because a common factor e^{-m}
// cancels between z and l. This keeps the rescale (which must wait for the
// previous z += P V) off the common path.
//
// Key blocks that are fully masked (past the causal diagonal, past the valid
// length) are never loaded: they are the empty summary.
//
// Schedule. A unit is one tile pair of one (batch item, head), or a single
// tile. With no more units than SMs every CTA takes one unit. Otherwise the
// host estimates, from the per-unit block counts (causal diagonal, valid
// lengths), one CTA per unit (handed out by the hardware in order) and one
// persistent CTA per SM that walks a fixed list of units (rounds of one unit
// per CTA, the CTA order reversed on odd rounds), each with the units pair
// by pair within a head or with the heavy causal pairs of all heads first
// (when the K and V to be read stay in L2), and launches the fastest;
// without a mask the pairs of a last, partly filled round may run as single
// tiles. In a persistent CTA the barrier phases run on from unit to unit: a
// unit's Q waits for the last S of the unit that used its Q buffer before
// (q_empty; at d_h = 64 there are two buffers, so the next unit's Q loads
// while the current unit runs), its first z = P V for the epilogue to read
// the current z out (o_empty), and its K/V loads and first S overlap the
// current unit's last blocks and epilogue.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <functional>
#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "internal.h"

namespace mha {
namespace {

constexpr int BLK_M = 128;  // query rows per tile (two tiles per CTA)
constexpr int BLK_N = 128;  // keys per block
constexpr int NTHREADS = 384;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;  // raise m only when the max grows by > 2^8

struct AttnTcParams {
  CUtensorMap qmap;  // Q: dims {d_h, n_q, B*h}, box {64, 128, 1}
  CUtensorMap kmap;  // K: dims {d_h, n_k, B*h}, box {64, 128, 1}
  CUtensorMap vmap;  // V: dims {d_vh, n_k, B*h}, box {64, 128, 1}
  void* Z;
  int n_q, n_k, h;
  int dv;            // d_vh: columns of z written per head (DV of the kernel or fewer)
  int npair;         // 256-row query tile pairs per (batch item, head)
  int units;         // units of work: pair_units pairs, then single tiles
  int pair_units;    // the first pair_units units are tile pairs; each later
                     // pair of the order is split into two single-tile units
  int nbh;           // h * B
  int pi_major;      // units ordered by tile pair first (heavy causal pairs of every head first)
  float cl2;         // |c| * log2(e)
  int negate;        // c < 0: S is computed as -Q K^T (MMA negate-A bit)
  int causal, padding, pad_queries;
  int32_t* err;
  uint64_t limit_ns;
  // Split over the keys (nsplit > 1): unit idx is split idx % nsplit of tile
  // pair idx / nsplit and folds key blocks [split * split_blocks, ...) only;
  // its summary goes to `part` and the last split of a tile to finish merges
  // them (`split_cnt` counts the published splits of each tile).
  int nsplit, split_blocks;
  float* part;      // [pair][tile][split] slots of (DV + 2) x 128 floats
  int* split_cnt;   // [pair][tile], zero on entry, left zero on exit
  int valid_len[MHA_MAX_PADDED_BATCH];
  int has_gate;                          // head_gate holds h entries (h <= MHA_MAX_GATED_HEADS)
  float head_gate[MHA_MAX_GATED_HEADS];  // per-head output scale, read only when has_gate
};

// bytes after the K/V ring: barriers (up to 64 x 8 B)
constexpr int EXTRA = 512;

template <int DQK, int DV>
struct ACfg {
  static constexpr int D_QK = DQK, D_V = DV;
  static constexpr int Q_TILE_BYTES = BLK_M * DQK * 2;
  static constexpr int K_BYTES = BLK_N * DQK * 2;
  static constexpr int V_BYTES = BLK_N * DV * 2;
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
  // epilogue staging: each of the 8 softmax warps, 16 rows of DV bf16
  static constexpr int STAGING = 8 * 16 * DV * 2;
  static constexpr int BUDGET = 227 * 1024 - 2 * Q_TILE_BYTES - 1024 - EXTRA - STAGING;
  static constexpr int STAGES = (BUDGET / STAGE_BYTES) > 4 ? 4 : (BUDGET / STAGE_BYTES);
  static constexpr int Q_BUFS = 1;  // Q tile pairs in shared memory
  static constexpr int SMEM = 2 * Q_TILE_BYTES + STAGES * STAGE_BYTES + 1024 + EXTRA + STAGING;
  // TMEM columns: S of tile 0 and 1, then z (O) of tile 0 and 1.
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + DV;
  static_assert(STAGES >= 2, "shared memory");
  static_assert(256 + 2 * DV <= TMEM_COLS, "tensor memory");
};

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if (globaltimer_ns() - t0 > 100000000ull) return;
  }
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum of 64 values as a tree of three-input maxima (depth 4).
__device__ __forceinline__ float max64(const uint32_t (&v)[64]) {
  float a[22], b[8];
#pragma unroll
  for (int i = 0; i < 21; ++i)
    a[i] = max3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]),
                __uint_as_float(v[3 * i + 2]));
  a[21] = __uint_as_float(v[63]);
#pragma unroll
  for (int i = 0; i < 7; ++i) b[i] = max3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[7] = a[21];
  return max3(max3(b[0], b[1], b[2]), max3(b[3], b[4], b[5]), fmaxf(b[6], b[7]));
}

// Number of 128-key blocks a tile starting at row tq0 must fold (0 when all
// its rows are padding).
__device__ __forceinline__ int tile_blocks(const AttnTcParams& P, int tq0, int L, int q_end) {
  if (tq0 >= q_end) return 0;
  int k_end = L;
  if (P.causal) k_end = min(k_end, tq0 + BLK_M);
  return (k_end + BLK_N - 1) / BLK_N;
}

// One unit of work: the 128-row query tile starting at q0 of (b, head) and,
// for a pair unit, the tile after it; with a split over the keys, only the
// key blocks [kb0, kb0 + nmax) of them.
struct Unit {
  int q0, head, b, L, q_end;
  int nb0, nb1, nmax;  // key blocks of tile 0, of tile 1, and the larger
  bool pair;           // tile 1 belongs to this unit (its rows are written here)
  bool has0, has1;     // the tile has rows to compute (some key blocks in all)
  int kb0;             // first key block of the unit
  int split, pidx;     // split number and tile pair index (split summaries)
};

// Tile pairs are ordered pair-fastest within each (batch item, head), or,
// with pi_major, (batch item, head)-fastest within each pair index; under a
// causal mask the heavy pairs (large q0) come first either way. Unit idx is
// pair idx while idx < pair_units; after that, units pair_units + 2 j and
// pair_units + 2 j + 1 are the two tiles of pair pair_units + j, on their own.
// With a split over the keys every unit is a pair: unit idx is split
// idx % nsplit of pair idx / nsplit.
__host__ __device__ inline void unit_coords(const AttnTcParams& P, int nsplit, int idx, int& pi,
                                            int& bh, int& tile, bool& pair, int& split,
                                            int& pidx) {
  pidx = idx;
  tile = 0;
  split = 0;
  pair = true;
  if (nsplit > 1) {
    pidx = idx / nsplit;
    split = idx % nsplit;
  } else if (idx >= P.pair_units) {
    const int j = idx - P.pair_units;
    pidx = P.pair_units + j / 2;
    tile = j & 1;
    pair = false;
  }
  pi = P.pi_major ? pidx / P.nbh : pidx % P.npair;
  bh = P.pi_major ? pidx % P.nbh : pidx / P.npair;
  if (P.causal) pi = P.npair - 1 - pi;
}

// Blocks [kb0, kb0 + n) of a tile with nb blocks in all that fall in split s.
__host__ __device__ inline int split_range(const AttnTcParams& P, int nsplit, int nb, int s,
                                           int& kb0) {
  if (nsplit <= 1) {
    kb0 = 0;
    return nb;
  }
  kb0 = s * P.split_blocks;
  const int n = nb - kb0;
  return n < 0 ? 0 : (n > P.split_blocks ? P.split_blocks : n);
}

// SPLIT: the kernel was launched for a split over the keys (P.nsplit > 1);
// without it every unit folds all of its key blocks.
template <bool SPLIT>
__device__ __forceinline__ Unit unit_at(const AttnTcParams& P, int idx) {
  Unit u;
  int pi, bh, tile;
  const int nsplit = SPLIT ? P.nsplit : 1;
  unit_coords(P, nsplit, idx, pi, bh, tile, u.pair, u.split, u.pidx);
  u.head = bh % P.h;
  u.b = bh / P.h;
  u.q0 = pi * 2 * BLK_M + tile * BLK_M;
  u.L = P.padding ? P.valid_len[u.b] : P.n_k;
  u.q_end = P.pad_queries ? min(u.L, P.n_q) : P.n_q;
  const int f0 = tile_blocks(P, u.q0, u.L, u.q_end);
  const int f1 = (u.pair && u.q0 + BLK_M < P.n_q) ? tile_blocks(P, u.q0 + BLK_M, u.L, u.q_end) : 0;
  u.has0 = f0 > 0;
  u.has1 = f1 > 0;
  u.nb0 = split_range(P, nsplit, f0, u.split, u.kb0);
  u.nb1 = split_range(P, nsplit, f1, u.split, u.kb0);
  u.nmax = u.nb1 > u.nb0 ? u.nb1 : u.nb0;  // tile 0's blocks are a prefix of tile 1's
  return u;
}

// The i-th unit of CTA c of G, or -1 past the end. Round i hands units
// [i G, i G + G) to the G CTAs, in reverse CTA order on odd rounds, so a CTA
// that drew a heavy causal pair in one round draws a light one in the next.
// With as many CTAs as units every CTA takes exactly its own unit.
__host__ __device__ inline int unit_index_of(const AttnTcParams& P, int G, int c, int i) {
  const int idx = i * G + ((i & 1) ? G - 1 - c : c);
  return idx < P.units ? idx : -1;
}

__device__ __forceinline__ int unit_index(const AttnTcParams& P, int i) {
  return unit_index_of(P, gridDim.x, blockIdx.x, i);
}

// The shared-memory ring and barriers a TMA producer thread fills.
struct Ring {
  uint8_t* q_s;        // Q_BUFS x the two Q tiles (unit i uses buffer i % Q_BUFS)
  uint8_t* kv_s;       // STAGES x (K block, V block)
  uint64_t* q_full;    // [Q_BUFS] Q tiles of a unit landed
  uint64_t* q_empty;   // [Q_BUFS] both tiles' S of the unit done with Q
  uint64_t* k_full;    // [STAGES]
  uint64_t* v_full;    // [STAGES]
  uint64_t* k_empty;   // [STAGES]
  uint64_t* v_empty;   // [STAGES]
};

// TMA producer thread of a persistent attention CTA. is_k: Q and the K blocks
// (warp 0), else the V blocks (warp 2), unit after unit through the same
// STAGES-deep ring (the ring position `it` runs on across units, so the next
// unit's first blocks load while the current unit's last ones are still
// being used).
template <class C, bool SPLIT>
__device__ __forceinline__ void produce(const AttnTcParams& P, const Ring& R, bool is_k,
                                        const WaitCtl& w) {
  const CUtensorMap* map = is_k ? &P.kmap : &P.vmap;
  uint64_t* full = is_k ? R.k_full : R.v_full;
  uint64_t* empty = is_k ? R.k_empty : R.v_empty;
  const int panels = is_k ? C::D_QK / 64 : C::D_V / 64;
  const uint32_t bytes = is_k ? C::K_BYTES : C::V_BYTES;
  tma_prefetch_desc(map);
  if (is_k) tma_prefetch_desc(&P.qmap);
  uint32_t it = 0;  // ring position
  int ui = 0;       // units loaded so far
  bool gave_up = false;
  int q_last = -1;  // unit number of this thread's last Q load
  for (int i = 0; !gave_up; ++i) {
    const int idx = unit_index(P, i);
    if (idx < 0) break;
    const Unit u = unit_at<SPLIT>(P, idx);
    if (u.nmax == 0) continue;  // all rows padding: nothing to load
    const int bh = u.b * P.h + u.head;
    if (is_k) {
      // the S MMAs of the unit that last used this Q buffer must be done
      const int qb = ui % C::Q_BUFS;
      if (ui >= C::Q_BUFS && !mbar_wait(R.q_empty + qb, (ui / C::Q_BUFS - 1) & 1, w)) {
        gave_up = true;
        break;
      }
      const int ntiles = u.nb1 > 0 ? 2 : 1;
      uint8_t* q_dst = R.q_s + qb * 2 * C::Q_TILE_BYTES;
      mbar_arrive_expect_tx(R.q_full + qb, ntiles * C::Q_TILE_BYTES);
      for (int t = 0; t < ntiles; ++t)
#pragma unroll
        for (int p = 0; p < C::D_QK / 64; ++p)
          tma_load_3d(q_dst + t * C::Q_TILE_BYTES + p * 16384, &P.qmap, R.q_full + qb, 64 * p,
                      u.q0 + t * BLK_M, bh);
      q_last = ui;
    }
    for (int kb = 0; kb < u.nmax; ++kb, ++it) {
      const int s = it % C::STAGES;
      uint8_t* dst = R.kv_s + s * C::STAGE_BYTES + (is_k ? 0 : C::K_BYTES);
      if (it >= (uint32_t)C::STAGES &&
          !mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1, w)) {
        gave_up = true;
        break;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
      for (int p = 0; p < panels; ++p)
        tma_load_3d(dst + p * 16384, map, &full[s], 64 * p, (u.kb0 + kb) * BLK_N, bh);
    }
    ++ui;
  }
  if (gave_up) {  // let this thread's loads land before the CTA exits
    if (is_k)
      for (int k = q_last - C::Q_BUFS + 1; k <= q_last; ++k)
        if (k >= 0) drain(R.q_full + k % C::Q_BUFS, (k / C::Q_BUFS) & 1);
    for (uint32_t k = (it > (uint32_t)C::STAGES ? it - C::STAGES : 0); k < it; ++k)
      drain(&full[k % C::STAGES], (k / C::STAGES) & 1);
  }
}

// ---------------------------------------------------------------------------
// Split over the keys: the summary of a split is published in a slot of its
// own, (pair, tile, split): z column-major (column c of row r at c * 128 + r,
// DV columns), then m[128] and l[128] (m in the scaled base-2 units of the
// kernel, -inf for a split without a key block of the tile: the empty
// summary). The thread block that publishes a tile's last split merges all
// of the tile's summaries with the merge of the Definition (m' = max m_s,
// l' = sum e^{m_s - m'} l_s, z' likewise) and writes z' / l' to Z. Nothing
// waits on another thread block: the last one to arrive finds every other
// summary already written.
// ---------------------------------------------------------------------------

template <int DV>
__device__ __forceinline__ float* split_slot(const AttnTcParams& P, int pidx, int t, int s) {
  return P.part + ((size_t)(pidx * 2 + t) * P.nsplit + s) * (size_t)((DV + 2) * BLK_M);
}

template <int NTHR>
__device__ __forceinline__ void tile_sync(int bar_id) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(NTHR) : "memory");
}

// Called by the NTHR threads that hold tile t's rows (named barrier bar_id)
// once the thread's NC columns [c0, c0 + NC) of row r of z are in the slot:
// publishes (m, l) of row r, counts the split, and in the last thread block
// merges and stores those columns of row r of Z. flag: one shared int.
template <int DV, int NC, int NTHR>
__device__ void split_finish(const AttnTcParams& P, const Unit& u, int t, int r, int c0,
                             float m, float l, int bar_id, volatile int* flag) {
  float* slot = split_slot<DV>(P, u.pidx, t, u.split);
  if (c0 == 0) {
    __stcg(slot + DV * BLK_M + r, m);
    __stcg(slot + (DV + 1) * BLK_M + r, l);
  }
  __threadfence();
  tile_sync<NTHR>(bar_id);
  if (r == 0 && c0 == 0) {
    int* cnt = P.split_cnt + u.pidx * 2 + t;
    const int last = atomicAdd(cnt, 1) == P.nsplit - 1;
    if (last) atomicExch(cnt, 0);  // every split has counted: ready for the next call
    __threadfence();
    *flag = last;
  }
  tile_sync<NTHR>(bar_id);
  if (!*flag) return;
  __threadfence();
  const int q = u.q0 + t * BLK_M + r;
  if (q >= P.n_q) return;
  const float* base = P.part + (size_t)(u.pidx * 2 + t) * P.nsplit * (size_t)((DV + 2) * BLK_M);
  constexpr size_t SLOT = (size_t)(DV + 2) * BLK_M;
  float M = -INFINITY;
  for (int s = 0; s < P.nsplit; ++s) M = fmaxf(M, __ldcg(base + s * SLOT + DV * BLK_M + r));
  float lsum = 0.f;
  for (int s = 0; s < P.nsplit; ++s) {
    const float ms = __ldcg(base + s * SLOT + DV * BLK_M + r);
    if (ms != -INFINITY) lsum += exp2f(ms - M) * __ldcg(base + s * SLOT + (DV + 1) * BLK_M + r);
  }
  const bool computed = q < u.q_end;
  const float inv = computed ? (P.has_gate ? P.head_gate[u.head] : 1.f) / lsum : 0.f;
  __nv_bfloat16* zrow = static_cast<__nv_bfloat16*>(P.Z) +
                        ((long long)u.b * P.n_q + q) * ((long long)P.h * P.dv) +
                        (long long)u.head * P.dv + c0;
#pragma unroll 1
  for (int cb = 0; cb < NC / 32; ++cb) {
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    if (computed) {
      for (int s = 0; s < P.nsplit; ++s) {
        const float ms = __ldcg(base + s * SLOT + DV * BLK_M + r);
        if (ms == -INFINITY) continue;  // the empty summary: the merge's identity
        const float ws = exp2f(ms - M);
        const float* zs = base + s * SLOT + (size_t)(c0 + 32 * cb) * BLK_M + r;
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = fmaf(ws, __ldcg(zs + j * BLK_M), acc[j]);
      }
    }
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(acc[2 * j] * inv, acc[2 * j + 1] * inv);
    uint4* dst = reinterpret_cast<uint4*>(zrow + 32 * cb);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c0 + 32 * cb + 8 * j < P.dv)
        dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
  }
}

// Epilogue stores through a warp's staging area in shared memory: its 16
// rows of a tile, DV bf16 columns each (row rho at rho DV / 8 16-byte
// chunks; chunk c at position c ^ (rho % 8), so that neither the lanes'
// writes of their own rows nor the row-wise reads meet on a bank). Each lane
// first stages the chunks of its half row; each store instruction then
// writes 32 / (DV / 8) whole rows of the head's columns, contiguous in Z.
template <int DV>
__device__ __forceinline__ void stage_chunk(uint4* st, int rho, int c, uint4 v) {
  st[rho * (DV / 8) + (c ^ (rho & 7))] = v;
}

// Stores the warp's staged rows q0w + rho (rho < 16) below n_q, columns below
// dv; zrow0: the head's first column in row q0w of Z.
template <int DV>
__device__ __forceinline__ void store_staged_rows(const uint4* st, __nv_bfloat16* zrow0,
                                                  long long row_stride, int q0w, int n_q,
                                                  int dv, int lane) {
  constexpr int CPR = DV / 8;     // chunks per row
  constexpr int RPI = 32 / CPR;   // rows per store instruction
  const int c = lane % CPR;
#pragma unroll
  for (int it = 0; it < 16 / RPI; ++it) {
    const int rho = it * RPI + lane / CPR;
    if (q0w + rho < n_q && 8 * c < dv)
      *reinterpret_cast<uint4*>(zrow0 + (long long)rho * row_stride + 8 * c) =
          st[rho * CPR + (c ^ (rho & 7))];
  }
}

template <int DQK, int DV, bool SPLIT>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_tc_kernel(const __grid_constant__ AttnTcParams P) {
  using C = ACfg<DQK, DV>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __nv_bfloat16* Zg = static_cast<__nv_bfloat16*>(P.Z);
  const long long zrow_stride = (long long)P.h * P.dv;  // d_vh <= DV columns per head

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_s = smem;  // two Q tiles
  uint8_t* kv_s = smem + 2 * C::Q_TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(kv_s + C::STAGES * C::STAGE_BYTES);
  uint64_t* q_full = bars;                  // Q tiles of the current unit landed
  uint64_t* q_empty = q_full + 1;           // both tiles' S of the unit done with Q
  uint64_t* k_full = q_empty + 1;           // [STAGES]
  uint64_t* v_full = k_full + C::STAGES;    // [STAGES]
  uint64_t* k_empty = v_full + C::STAGES;   // [STAGES] freed once S of both tiles is done
  uint64_t* v_empty = k_empty + C::STAGES;  // [STAGES] freed once both z += P V are done
  uint64_t* s_full = v_empty + C::STAGES;   // [2] per tile
  uint64_t* p_full = s_full + 2;            // [2] per tile
  uint64_t* o_full = p_full + 2;            // [2] per tile
  uint64_t* o_empty = o_full + 2;           // [2] per tile: z read out by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint4* staging = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(bars) + EXTRA);
  volatile int* split_flag = abort_flag + 1;  // the last split of a tile merges

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 2);  // one arrival per MMA issuer
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 2);  // one arrival per tile (issuer)
      mbar_init(&v_empty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 8);   // one arrival per softmax warp
      mbar_init(&o_full[t], 1);
      mbar_init(&o_empty[t], 8);  // one arrival per softmax warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The prologue above touched only this CTA's shared and tensor memory. The
  // next kernel may start its own now; this one reads its inputs and writes
  // its outputs only once the previous kernel has completed.
  grid_dep_launch_dependents();
  grid_dep_wait();
  const WaitCtl w{P.err, abort_flag, P.limit_ns};
  const Ring ring{q_s, kv_s, q_full, q_empty, k_full, v_full, k_empty, v_empty};

  if (warp < 4) {
    if ((warp == 0 || warp == 2) && lane == 0) {
      produce<C, SPLIT>(P, ring, warp == 0, w);
    } else if ((warp == 1 || warp == 3) && lane == 0) {
      // Two MMA issuers, one per query tile (warp 1: tile 0, warp 3: tile 1).
      // Each keeps its own short tensor-instruction queue filled, so the
      // bookkeeping of one (barrier waits, commits) is covered by the other's
      // queued MMAs. Within a tile the order S_j, P_j V_j, S_{j+1}, ... is kept
      // by the single issuing thread (S_{j+1} overwrites P_j in TMEM); the
      // next unit's first S follows the current unit's last P V the same way,
      // so it runs while the softmax warps write the current unit out.
      const int t = warp == 1 ? 0 : 1;
      const uint32_t idesc_qk =
          idesc_bf16_f32(BLK_M, BLK_N, 0, 0) | (P.negate ? (1u << 13) : 0u);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BLK_M, DV, 0, 1);
      // Shared-memory descriptors are built once; each operand is a base
      // descriptor plus a small constant (the start address sits in the low
      // 14 bits and every shared address is below 256 KB).
      const uint64_t qd = sdesc_sw128(smem_u32(q_s + t * C::Q_TILE_BYTES), 16, 1024);
      const uint64_t k_desc = sdesc_sw128(smem_u32(kv_s), 16, 1024);
      const uint64_t v_desc = sdesc_sw128(smem_u32(kv_s + C::K_BYTES), 16384, 1024);
      constexpr uint64_t STAGE_D = C::STAGE_BYTES >> 4;
      const uint32_t s_tmem = tmem + (t ? C::S_COL1 : C::S_COL0);
      const uint32_t o_tmem = tmem + (t ? C::O_COL1 : C::O_COL0);
      // r: ring position of the K/V block
      auto issue_s = [&](uint32_t r) {
        const uint64_t kd = k_desc + (uint64_t)(r % C::STAGES) * STAGE_D;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          // 16 elements = 32 B inside a 128 B swizzle row; 64-element panels 16 KB apart
          const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
          umma_ss(s_tmem, qd + off, kd + off, idesc_qk, kk > 0);
        }
        umma_commit(&s_full[t]);
        umma_commit(&k_empty[r % C::STAGES]);  // this tile is done with this K block
      };
      auto issue_pv = [&](uint32_t r, bool first) {
        const uint64_t vd = v_desc + (uint64_t)(r % C::STAGES) * STAGE_D;
#pragma unroll
        for (int kk = 0; kk < BLK_N / 16; ++kk) {
          // V is MN-major: 16 key rows of 128 B; 64-column panels 16 KB apart
          umma_ts(o_tmem, s_tmem + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                  (!first || kk > 0));
        }
        umma_commit(&o_full[t]);
        umma_commit(&v_empty[r % C::STAGES]);  // this tile is done with this V block
      };
      uint32_t base = 0;  // ring position of the current unit's block 0
      uint32_t c = 0;     // blocks of this tile folded so far (s/p/o_full phases)
      uint32_t act = 0;   // units in which this tile had rows to compute
      int ui = 0;
      bool ok = true;
      bool inflight = false;  // MMAs of this thread may still be running
      for (int i = 0; ok; ++i) {
        const int idx = unit_index(P, i);
        if (idx < 0) break;
        const Unit u = unit_at<SPLIT>(P, idx);
        if (u.nmax == 0) continue;
        const int nbt = t ? u.nb1 : u.nb0;
        // the unit's Q tiles are in (this also orders the q_empty arrival
        // below after the previous unit's phase)
        if (!mbar_wait(q_full, ui & 1, w)) {
          ok = false;
          break;
        }
        if (nbt > 0) {
          if (!mbar_wait(&k_full[base % C::STAGES], (base / C::STAGES) & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(base);
          inflight = true;
          if (nbt == 1) umma_commit(q_empty);  // the unit's last S is issued
          for (int kb = 0; kb < nbt; ++kb, ++c) {
            const uint32_t r = base + kb;
            const int s = r % C::STAGES;
            if (!mbar_wait(&v_full[s], (r / C::STAGES) & 1, w) ||
                !mbar_wait(&p_full[t], c & 1, w)) {
              ok = false;
              break;
            }
            // the previous unit's z must have been read out before the first
            // z = P V of this unit overwrites it
            if (kb == 0 && act > 0 && !mbar_wait(&o_empty[t], (act - 1) & 1, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(r, kb == 0);
            if (kb + 1 < nbt) {
              if (!mbar_wait(&k_full[(r + 1) % C::STAGES], ((r + 1) / C::STAGES) & 1, w)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(r + 1);  // after P_kb V_kb in this thread's order
              if (kb + 2 == nbt) umma_commit(q_empty);  // the unit's last S is issued
            }
          }
          if (!ok) break;
          ++act;
        } else {
          mbar_arrive(q_empty);  // this tile has no rows in the unit: no S reads Q
        }
        // A tile with fewer blocks than the unit (causal tile 0, or a padding
        // tile 1) still releases the remaining K/V stages, each once that
        // block's data is in (so the arrival lands in that block's phase of
        // the empty barrier).
        for (int k2 = nbt; k2 < u.nmax && ok; ++k2) {
          const uint32_t r = base + k2;
          const int s = r % C::STAGES;
          const uint32_t par = (r / C::STAGES) & 1;
          if (!mbar_wait(&k_full[s], par, w)) {
            ok = false;
            break;
          }
          mbar_arrive(&k_empty[s]);
          if (!mbar_wait(&v_full[s], par, w)) {
            ok = false;
            break;
          }
          mbar_arrive(&v_empty[s]);
        }
        base += u.nmax;
        ++ui;
      }
      if (!ok && inflight) {  // gave up: wait for this thread's MMAs before TMEM is released
        umma_commit(&s_full[t]);
        drain(&s_full[t], 0);
        drain(&s_full[t], 1);
      }
    }
  } else {
    // Softmax: warps 4..11 take tile 0 then tile 1 for every key block, so
    // the two tiles' softmaxes alternate (they share the exponential units)
    // and each overlaps the other tile's MMAs. A warp holds 16 rows, lanes i
    // and i + 16 the two halves of row 32 g + 16 hh + i (`half` = lane / 16:
    // key columns [64 half, 64 half + 64) of S, value columns
    // [half DV/2, (half + 1) DV/2) of z), read and written with the
    // half-split TMEM shape; the partners combine their partial row maximum
    // with a shuffle and keep partial row sums, added once at the end of a
    // unit. Both halves of a row come in with the same load, so P may
    // overwrite the first columns of S as soon as that load is waited for.
    const int g = warp & 3;            // TMEM lane slice 32*g .. 32*g+31
    const int hh = (warp - 4) >> 2;    // 0: lanes 32g .. 32g+15, 1: lanes 32g+16 .. 32g+31
    const int half = lane >> 4;
    const int r = 32 * g + 16 * hh + (lane & 15);
    const uint32_t lane_off = static_cast<uint32_t>(32 * g + 16 * hh) << 16;
    const float cl2 = P.cl2;
    const float2 cl2x2 = make_float2(cl2, cl2);
    uint32_t c[2] = {0, 0};  // blocks folded per tile so far (s/p/o_full phases)
    bool ok = true;
    for (int i = 0;; ++i) {
      const int idx = unit_index(P, i);
      if (idx < 0) break;
      const Unit u = unit_at<SPLIT>(P, idx);
      const long long zbase = (long long)u.b * P.n_q * zrow_stride + (long long)u.head * P.dv;
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      for (int kb = 0; kb < u.nmax; ++kb) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nblk = t ? u.nb1 : u.nb0;
          if (kb >= nblk) continue;  // uniform across the warp
          const int tq0 = u.q0 + t * BLK_M;
          const int q = tq0 + r;
          const uint32_t s_addr = tmem + lane_off + (t ? C::S_COL1 : C::S_COL0);
          const uint32_t o_addr = tmem + lane_off + (t ? C::O_COL1 : C::O_COL0);
          const uint32_t cc = c[t]++;
          if (ok && !mbar_wait(&s_full[t], cc & 1, w)) ok = false;
          if (!__all_sync(0xffffffffu, ok)) {  // do no work
            ok = false;
            continue;
          }
          tc_fence_after();
          const int k0 = (u.kb0 + kb) * BLK_N;
          const bool masked = (k0 + BLK_N > u.L) || (P.causal && k0 + BLK_N - 1 > tq0);
          // allowed keys of this row in this block: k0 + c < lim
          const int lim = (masked ? (P.causal ? min(u.L, q + 1) : u.L) - k0 : BLK_N) - 64 * half;
          uint32_t sr[64];
          tmem_ld_x2_64<64>(s_addr, sr);
          tmem_wait_ld();
          if (masked) {
            // forbidden keys get s = -inf, hence weight 2^{-inf} = 0 exactly
            // (the scale cl2 is positive, never 0); blocks without forbidden
            // keys skip this branch
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (j >= lim) sr[j] = __float_as_uint(-INFINITY);
          }
          const float mh = max64(sr);
          const float mx = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 16));
          const float m_blk = (mx == -INFINITY) ? -INFINITY : mx * cl2;
          // raise the running max only past the threshold (or on the first block)
          const bool raise =
              (m_run[t] == -INFINITY) ? true : (m_blk > m_run[t] + RESCALE_LOG2);
          const float m_new = raise ? fmaxf(m_run[t], m_blk) : m_run[t];
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          const float alpha = ex2_approx(m_run[t] - m_use);  // e^{m - m'}: 1 when m is kept
          const float2 negm = make_float2(-m_use, -m_use);
          float2 sum = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
          // p = 2^{c log2(e) s - m} as bf16 over the first 64 columns of S:
          // this half's keys go to P columns [32 half, 32 half + 32)
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            float2 x0 = __ffma2_rn(
                make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])), cl2x2, negm);
            float2 x1 = __ffma2_rn(
                make_float2(__uint_as_float(sr[j + 2]), __uint_as_float(sr[j + 3])), cl2x2,
                negm);
            x0.x = ex2_approx(x0.x);
            x0.y = ex2_approx(x0.y);
            x1.x = ex2_approx(x1.x);
            x1.y = ex2_approx(x1.y);
            sum = __fadd2_rn(sum, x0);
            sum_b = __fadd2_rn(sum_b, x1);
            pk[j / 2] = pack_bf16x2(x0.x, x0.y);
            pk[j / 2 + 1] = pack_bf16x2(x1.x, x1.y);
          }
          tmem_st_x2_32<32>(s_addr, pk);
          l_run[t] = l_run[t] * alpha + ((sum.x + sum.y) + (sum_b.x + sum_b.y));
          // merge: rescale this row of z by e^{m - m'} when m was raised; z must
          // already hold every earlier block (wait for the previous z += P V)
          if (__any_sync(0xffffffffu, kb > 0 && raise)) {
            if (!__all_sync(0xffffffffu, mbar_wait(&o_full[t], (cc - 1) & 1, w))) {
              ok = false;
              continue;
            }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < DV / 64; ++cb) {
              uint32_t o[32];
              const uint32_t oa = o_addr + 32 * cb;
              tmem_ld_x2_32<DV / 2>(oa, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const float2 v = __fmul2_rn(
                    make_float2(__uint_as_float(o[j]), __uint_as_float(o[j + 1])),
                    make_float2(alpha, alpha));
                o[j] = __float_as_uint(v.x);
                o[j + 1] = __float_as_uint(v.y);
              }
              tmem_st_x2_32<DV / 2>(oa, o);
            }
          }
          m_run[t] = m_new;
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[t]);
        }
      }
      // Epilogue of the unit: z / l for this half of each row, in the
      // concatenated layout; then z of the tile is free for the next unit.
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t == 1 && !u.pair) continue;  // those rows are another unit's
        const int nblk = t ? u.nb1 : u.nb0;
        const int q = u.q0 + t * BLK_M + r;
        const uint32_t o_addr = tmem + lane_off + (t ? C::O_COL1 : C::O_COL0);
        __nv_bfloat16* zrow = Zg + zbase + (long long)q * zrow_stride + half * (DV / 2);
        if (SPLIT ? !(t ? u.has1 : u.has0) : nblk == 0) {
          // the whole tile is padding: its rows are zero (written by split 0)
          if (q < P.n_q && u.split == 0) {
#pragma unroll
            for (int j = 0; j < DV / 16; ++j)
              if (half * (DV / 2) + 8 * j < P.dv)
                reinterpret_cast<uint4*>(zrow)[j] = make_uint4(0, 0, 0, 0);
          }
          continue;
        }
        // the row sum is the two partners' partial sums (same running max)
        const float l_tot = l_run[t] + __shfl_xor_sync(0xffffffffu, l_run[t], 16);
        if (SPLIT) {
          // publish this split's summary of the tile's rows (the empty
          // summary when the split holds none of its key blocks)
          float m_s = -INFINITY, l_s = 0.f;
          if (nblk > 0) {
            l_s = l_tot;
            m_s = m_run[t];
            if (ok && !__all_sync(0xffffffffu, mbar_wait(&o_full[t], (c[t] - 1) & 1, w)))
              ok = false;
            if (ok) {
              tc_fence_after();
              float* zs = split_slot<DV>(P, u.pidx, t, u.split) + (half * (DV / 2)) * BLK_M + r;
#pragma unroll
              for (int cb = 0; cb < DV / 64; ++cb) {
                uint32_t o[32];
                tmem_ld_x2_32<DV / 2>(o_addr + 32 * cb, o);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) __stcg(zs + (32 * cb + j) * BLK_M, __uint_as_float(o[j]));
              }
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&o_empty[t]);
            }
          }
          split_finish<DV, DV / 2, 256>(P, u, t, r, half * (DV / 2), m_s, l_s, 9, split_flag);
          continue;
        }
        if (!ok || !__all_sync(0xffffffffu, mbar_wait(&o_full[t], (c[t] - 1) & 1, w))) {
          ok = false;
          continue;
        }
        tc_fence_after();
        const bool computed = q < u.q_end;
        const float inv = computed ? (P.has_gate ? P.head_gate[u.head] : 1.f) / l_tot : 0.f;
        uint4* st = staging + (warp - 4) * (16 * DV / 8);
#pragma unroll
        for (int cb = 0; cb < DV / 64; ++cb) {
          uint32_t o[32];
          tmem_ld_x2_32<DV / 2>(o_addr + 32 * cb, o);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = computed ? pack_bf16x2(__uint_as_float(o[2 * j]) * inv,
                                           __uint_as_float(o[2 * j + 1]) * inv)
                             : 0u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            stage_chunk<DV>(st, lane & 15, (half * (DV / 2) + 32 * cb) / 8 + j,
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_empty[t]);  // z is read: the next unit may overwrite it
        // the warp's rows, row by row (columns past d_vh, read as zeros from
        // V, are not written)
        const int q0w = u.q0 + t * BLK_M + 32 * g + 16 * hh;
        store_staged_rows<DV>(st, Zg + zbase + (long long)q0w * zrow_stride, zrow_stride, q0w,
                              P.n_q, P.dv, lane);
        __syncwarp();  // the staging area is rewritten by the next tile
      }
    }
  }
  // Every lane of a warp meets here before the CTA-wide barrier: a barrier
  // counts whole warps, so a warp must not reach it split across branches.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Variant for d_vh = 64: S, P and z of both tiles in separate TMEM columns
// (S 2 x 128, P 2 x 64 as bf16 pairs, z 2 x 64 = 512). A tile's next S can
// then be computed as soon as its softmax warps have read the current S
// into registers (s_free), while they still work on it, instead of after the
// tile's P V; and each tile has its own eight softmax warps, so one tile's
// softmax latency (loads, exchange, barrier waits) overlaps the other's
// exponentials. P is overwritten only once the previous block's P V is done.
// ---------------------------------------------------------------------------

constexpr int SP_THREADS = 128 + 2 * 256;  // 4 control warps, 8 softmax warps per tile

template <int DQK>
struct SpCfg {
  static constexpr int D_QK = DQK, D_V = 64;
  static constexpr int Q_TILE_BYTES = BLK_M * DQK * 2;
  static constexpr int K_BYTES = BLK_N * DQK * 2;
  static constexpr int V_BYTES = BLK_N * 64 * 2;
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
  // barriers (up to 64 x 8 B)
  static constexpr int EXTRA_SP = 512;
  // epilogue staging: each of the 16 softmax warps, 16 rows of 64 bf16
  static constexpr int STAGING = 16 * 16 * 64 * 2;
  // a second pair of Q tiles (the next unit's, loaded while the current one
  // runs) where it leaves the ring at four stages
  static constexpr int Q_BUFS =
      (227 * 1024 - 4 * Q_TILE_BYTES - 1024 - EXTRA_SP - STAGING) / STAGE_BYTES >= 4 ? 2 : 1;
  static constexpr int BUDGET =
      227 * 1024 - 2 * Q_BUFS * Q_TILE_BYTES - 1024 - EXTRA_SP - STAGING;
  static constexpr int STAGES = (BUDGET / STAGE_BYTES) > 4 ? 4 : (BUDGET / STAGE_BYTES);
  static constexpr int SMEM =
      2 * Q_BUFS * Q_TILE_BYTES + STAGES * STAGE_BYTES + 1024 + EXTRA_SP + STAGING;
  // TMEM columns of tile t: S at 128 t, P at 256 + 64 t, z at 384 + 64 t
  static constexpr uint32_t S_COL = 0, P_COL = 256, O_COL = 384;
  static_assert(STAGES >= 2, "shared memory");
};

template <int DQK, bool SPLIT>
__global__ void __launch_bounds__(SP_THREADS, 1)
    attn_tc_sp_kernel(const __grid_constant__ AttnTcParams P) {
  using C = SpCfg<DQK>;
  constexpr int DV = 64;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __nv_bfloat16* Zg = static_cast<__nv_bfloat16*>(P.Z);
  const long long zrow_stride = (long long)P.h * P.dv;  // d_vh <= 64 columns per head

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + 2 * C::Q_BUFS * C::Q_TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(kv_s + C::STAGES * C::STAGE_BYTES);
  uint64_t* q_full = bars;                  // [Q_BUFS]
  uint64_t* q_empty = q_full + C::Q_BUFS;   // [Q_BUFS]
  uint64_t* k_full = q_empty + C::Q_BUFS;   // [STAGES]
  uint64_t* v_full = k_full + C::STAGES;    // [STAGES]
  uint64_t* k_empty = v_full + C::STAGES;   // [STAGES]
  uint64_t* v_empty = k_empty + C::STAGES;  // [STAGES]
  uint64_t* s_full = v_empty + C::STAGES;   // [2] S of the block is in TMEM
  uint64_t* s_free = s_full + 2;            // [2] the softmax warps have read S
  uint64_t* p_full = s_free + 2;            // [2] P of the block is in TMEM
  uint64_t* o_full = p_full + 2;            // [2] z += P V done
  uint64_t* o_empty = o_full + 2;           // [2] z read out by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint4* staging = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(bars) + C::EXTRA_SP);
  volatile int* split_flag = abort_flag + 1;  // [2]: the last split of a tile merges

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::Q_BUFS; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 2);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 2);
      mbar_init(&v_empty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 8);   // one arrival per softmax warp of the tile
      mbar_init(&p_full[t], 8);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_empty[t], 8);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_launch_dependents();
  grid_dep_wait();
  const WaitCtl w{P.err, abort_flag, P.limit_ns};
  const Ring ring{q_s, kv_s, q_full, q_empty, k_full, v_full, k_empty, v_empty};

  if (warp < 4) {
    if ((warp == 0 || warp == 2) && lane == 0) {
      produce<C, SPLIT>(P, ring, warp == 0, w);
    } else if ((warp == 1 || warp == 3) && lane == 0) {
      // MMA issuer of tile t. Order per tile: S_0, S_1 (once S_0 is read),
      // P_0 V, S_2 (once S_1 is read), P_1 V, ...; S_{j+1} does not wait for
      // P_j V because P has columns of its own.
      const int t = warp == 1 ? 0 : 1;
      const uint32_t idesc_qk =
          idesc_bf16_f32(BLK_M, BLK_N, 0, 0) | (P.negate ? (1u << 13) : 0u);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BLK_M, DV, 0, 1);
      const uint64_t qd0 = sdesc_sw128(smem_u32(q_s + t * C::Q_TILE_BYTES), 16, 1024);
      uint64_t qd = qd0;  // the current unit's Q buffer
      const uint64_t k_desc = sdesc_sw128(smem_u32(kv_s), 16, 1024);
      const uint64_t v_desc = sdesc_sw128(smem_u32(kv_s + C::K_BYTES), 16384, 1024);
      constexpr uint64_t STAGE_D = C::STAGE_BYTES >> 4;
      const uint32_t s_tmem = tmem + C::S_COL + 128 * t;
      const uint32_t p_tmem = tmem + C::P_COL + 64 * t;
      const uint32_t o_tmem = tmem + C::O_COL + 64 * t;
      auto issue_s = [&](uint32_t r) {
        const uint64_t kd = k_desc + (uint64_t)(r % C::STAGES) * STAGE_D;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
          umma_ss(s_tmem, qd + off, kd + off, idesc_qk, kk > 0);
        }
        umma_commit(&s_full[t]);
        umma_commit(&k_empty[r % C::STAGES]);
      };
      auto issue_pv = [&](uint32_t r, bool first) {
        const uint64_t vd = v_desc + (uint64_t)(r % C::STAGES) * STAGE_D;
#pragma unroll
        for (int kk = 0; kk < BLK_N / 16; ++kk)
          umma_ts(o_tmem, p_tmem + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                  (!first || kk > 0));
        umma_commit(&o_full[t]);
        umma_commit(&v_empty[r % C::STAGES]);
      };
      uint32_t base = 0;  // ring position of the current unit's block 0
      uint32_t cs = 0;    // S issued for this tile so far (s_full / s_free phases)
      uint32_t c = 0;     // P V issued for this tile so far (p_full / o_full phases)
      uint32_t act = 0;   // units in which this tile had rows to compute
      int ui = 0;
      bool ok = true, inflight = false;
      // S number cs may be issued once S number cs - 1 has been read out
      auto s_slot_free = [&]() { return cs == 0 || mbar_wait(&s_free[t], (cs - 1) & 1, w); };
      for (int i = 0; ok; ++i) {
        const int idx = unit_index(P, i);
        if (idx < 0) break;
        const Unit u = unit_at<SPLIT>(P, idx);
        if (u.nmax == 0) continue;
        const int nbt = t ? u.nb1 : u.nb0;
        const int qb = ui % C::Q_BUFS;
        qd = qd0 + (uint64_t)((qb * 2 * C::Q_TILE_BYTES) >> 4);
        if (!mbar_wait(q_full + qb, (ui / C::Q_BUFS) & 1, w)) {
          ok = false;
          break;
        }
        if (nbt > 0) {
          if (!s_slot_free() ||
              !mbar_wait(&k_full[base % C::STAGES], (base / C::STAGES) & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(base);
          ++cs;
          inflight = true;
          if (nbt == 1) umma_commit(q_empty + qb);  // the unit's last S is issued
          for (int kb = 0; kb < nbt; ++kb, ++c) {
            const uint32_t r = base + kb;
            if (kb + 1 < nbt) {
              if (!s_slot_free() ||
                  !mbar_wait(&k_full[(r + 1) % C::STAGES], ((r + 1) / C::STAGES) & 1, w)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(r + 1);
              ++cs;
              if (kb + 2 == nbt) umma_commit(q_empty + qb);
            }
            if (!mbar_wait(&v_full[r % C::STAGES], (r / C::STAGES) & 1, w) ||
                !mbar_wait(&p_full[t], c & 1, w) ||
                (kb == 0 && act > 0 && !mbar_wait(&o_empty[t], (act - 1) & 1, w))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(r, kb == 0);
          }
          if (!ok) break;
          ++act;
        } else {
          mbar_arrive(q_empty + qb);  // this tile has no rows in the unit: no S reads Q
        }
        for (int k2 = nbt; k2 < u.nmax && ok; ++k2) {
          const uint32_t r = base + k2;
          const int s = r % C::STAGES;
          const uint32_t par = (r / C::STAGES) & 1;
          if (!mbar_wait(&k_full[s], par, w)) {
            ok = false;
            break;
          }
          mbar_arrive(&k_empty[s]);
          if (!mbar_wait(&v_full[s], par, w)) {
            ok = false;
            break;
          }
          mbar_arrive(&v_empty[s]);
        }
        base += u.nmax;
        ++ui;
      }
      if (!ok && inflight) {  // gave up: wait for this thread's MMAs before TMEM is released
        umma_commit(&s_full[t]);
        drain(&s_full[t], 0);
        drain(&s_full[t], 1);
      }
    }
  } else {
    // Softmax: warps 4..11 own tile 0, warps 12..19 tile 1. A warp holds 16
    // rows of its tile, lanes i and i + 16 the two halves of row
    // 32 g + 16 hh + i (`half` = lane / 16: key columns [64 half, 64 half + 64)
    // of S, P columns [32 half, 32 half + 32), z columns [32 half,
    // 32 half + 32)), read and written with the half-split TMEM shape; the
    // partners combine their partial row maximum and row sum with a shuffle.
    const int t = (warp - 4) >> 3;
    const int hh = ((warp - 4) >> 2) & 1;
    const int g = warp & 3;  // TMEM lane slice 32*g .. 32*g+31
    const int half = lane >> 4;
    const int r = 32 * g + 16 * hh + (lane & 15);
    const uint32_t lane_off = static_cast<uint32_t>(32 * g + 16 * hh) << 16;
    const uint32_t s_addr = tmem + lane_off + C::S_COL + 128 * t;
    const uint32_t p_addr = tmem + lane_off + C::P_COL + 64 * t;
    const uint32_t o_addr = tmem + lane_off + C::O_COL + 64 * t;
    const float cl2 = P.cl2;
    const float2 cl2x2 = make_float2(cl2, cl2);
    uint32_t cS = 0;  // blocks of this tile folded so far (s_full / s_free / p_full / o_full)
    bool ok = true;
    for (int i = 0;; ++i) {
      const int idx = unit_index(P, i);
      if (idx < 0) break;
      const Unit u = unit_at<SPLIT>(P, idx);
      if (t == 1 && !u.pair) continue;  // a single-tile unit: those rows are another unit's
      const int nblk = t ? u.nb1 : u.nb0;
      const int tq0 = u.q0 + t * BLK_M;
      const int q = tq0 + r;
      float m_run = -INFINITY, l_run = 0.f;
      for (int kb = 0; kb < nblk; ++kb) {
        const uint32_t cc = cS++;
        if (ok && !mbar_wait(&s_full[t], cc & 1, w)) ok = false;
        if (!__all_sync(0xffffffffu, ok)) {  // do no work
          ok = false;
          continue;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld_x2_64<64>(s_addr, sr);
        tmem_wait_ld();
        // S is in registers: the tile's next S may be computed into its columns
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[t]);
        const int k0 = (u.kb0 + kb) * BLK_N;
        const bool masked = (k0 + BLK_N > u.L) || (P.causal && k0 + BLK_N - 1 > tq0);
        const int lim = (masked ? (P.causal ? min(u.L, q + 1) : u.L) - k0 : BLK_N) - 64 * half;
        if (masked) {
          // forbidden keys get s = -inf, hence weight 2^{-inf} = 0 exactly
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (j >= lim) sr[j] = __float_as_uint(-INFINITY);
        }
        const float mh = max64(sr);
        const float mx = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 16));
        const float m_blk = (mx == -INFINITY) ? -INFINITY : mx * cl2;
        // raise the running max only past the threshold (or on the first block)
        const bool raise = (m_run == -INFINITY) ? true : (m_blk > m_run + RESCALE_LOG2);
        const float m_new = raise ? fmaxf(m_run, m_blk) : m_run;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m_run - m_use);  // e^{m - m'}: 1 when m is kept
        const float2 negm = make_float2(-m_use, -m_use);
        // p = 2^{c log2(e) s - m}, this half row of 64 into registers
        float2 sum = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          float2 x0 = __ffma2_rn(
              make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])), cl2x2, negm);
          float2 x1 = __ffma2_rn(
              make_float2(__uint_as_float(sr[j + 2]), __uint_as_float(sr[j + 3])), cl2x2, negm);
          x0.x = ex2_approx(x0.x);
          x0.y = ex2_approx(x0.y);
          x1.x = ex2_approx(x1.x);
          x1.y = ex2_approx(x1.y);
          sum = __fadd2_rn(sum, x0);
          sum_b = __fadd2_rn(sum_b, x1);
          pk[j / 2] = pack_bf16x2(x0.x, x0.y);
          pk[j / 2 + 1] = pack_bf16x2(x1.x, x1.y);
        }
        l_run = l_run * alpha + ((sum.x + sum.y) + (sum_b.x + sum_b.y));
        // the previous block's z += P V must be done before P is overwritten
        // (and before z is rescaled); by now it normally is
        if (kb > 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(&o_full[t], (cc - 1) & 1, w))) {
            ok = false;
            continue;
          }
          tc_fence_after();
        }
        tmem_st_x2_32<32>(p_addr, pk);
        if (__any_sync(0xffffffffu, kb > 0 && raise)) {
          // merge: rescale this half row of z by e^{m - m'}
          uint32_t o[32];
          tmem_ld_x2_32<32>(o_addr, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 v =
                __fmul2_rn(make_float2(__uint_as_float(o[j]), __uint_as_float(o[j + 1])),
                           make_float2(alpha, alpha));
            o[j] = __float_as_uint(v.x);
            o[j + 1] = __float_as_uint(v.y);
          }
          tmem_st_x2_32<32>(o_addr, o);
        }
        m_run = m_new;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
      }
      // Epilogue of the unit: z / l for this half of each row
      __nv_bfloat16* zrow = Zg + (long long)u.b * P.n_q * zrow_stride + (long long)u.head * P.dv +
                            (long long)q * zrow_stride + 32 * half;
      if (SPLIT ? !(t ? u.has1 : u.has0) : nblk == 0) {
        // the whole tile is padding: its rows are zero (written by split 0)
        if (q < P.n_q && u.split == 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (32 * half + 8 * j < P.dv)
              reinterpret_cast<uint4*>(zrow)[j] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      // the row sum is the two partners' partial sums (same running max)
      const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
      if (SPLIT) {
        // publish this split's summary of the tile's rows (the empty summary
        // when the split holds none of its key blocks)
        float m_s = -INFINITY, l_s = 0.f;
        if (nblk > 0) {
          l_s = l_tot;
          m_s = m_run;
          if (ok && !__all_sync(0xffffffffu, mbar_wait(&o_full[t], (cS - 1) & 1, w))) ok = false;
          if (ok) {
            tc_fence_after();
            uint32_t o[32];
            tmem_ld_x2_32<32>(o_addr, o);
            tmem_wait_ld();
            float* zs = split_slot<DV>(P, u.pidx, t, u.split) + (32 * half) * BLK_M + r;
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(zs + j * BLK_M, __uint_as_float(o[j]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[t]);
          }
        }
        split_finish<DV, 32, 256>(P, u, t, r, 32 * half, m_s, l_s, 9 + t, split_flag + t);
        continue;
      }
      if (!ok || !__all_sync(0xffffffffu, mbar_wait(&o_full[t], (cS - 1) & 1, w))) {
        ok = false;
        continue;
      }
      tc_fence_after();
      const bool computed = q < u.q_end;
      const float inv = computed ? (P.has_gate ? P.head_gate[u.head] : 1.f) / l_tot : 0.f;
      uint32_t o[32];
      tmem_ld_x2_32<32>(o_addr, o);
      tmem_wait_ld();
      uint4* st = staging + (warp - 4) * (16 * DV / 8);
      {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = computed ? pack_bf16x2(__uint_as_float(o[2 * j]) * inv,
                                         __uint_as_float(o[2 * j + 1]) * inv)
                           : 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          stage_chunk<DV>(st, lane & 15, 4 * half + j,
                          make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[t]);  // z is read: the next unit may overwrite it
      const int q0w = tq0 + r - (lane & 15);     // the warp's first row
      // (columns past d_vh, read as zeros from V, are not written)
      store_staged_rows<DV>(st, zrow - 32 * half - (long long)(lane & 15) * zrow_stride,
                            zrow_stride, q0w, P.n_q, P.dv, lane);
      __syncwarp();  // the staging area is rewritten by the next tile
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Host side of the schedule. The cost of a unit is counted in tile steps
// (one 128 x 128 block of one tile); each CTA also pays a fixed part per unit
// that it cannot overlap: in a CTA of its own, the start-up (loads, first S)
// and the epilogue, about UNIT_FIXED steps on GB300; in a persistent CTA only
// the epilogue, PERSIST_FIXED steps (the next unit's loads and first S run
// under the current unit's last steps).
constexpr int UNIT_FIXED = 5, PERSIST_FIXED = 2;
constexpr long long MAX_SIMULATED_UNITS = 1 << 16;
constexpr double PI_MAJOR_MAX_KV_BYTES = 112.0 * (1 << 20);  // K and V read, kept in L2

// A tile on its own cannot overlap its softmax with its MMAs: a step costs
// the softmax plus the MMAs, about 1 + 4 (d_h + d_vh) / 1600 pair steps.
// With a split over the keys a unit also publishes its summaries and may
// merge them, about SPLIT_FIXED steps.
constexpr double SPLIT_FIXED = 1.0;

double unit_cost_host(const AttnTcParams& P, int idx, double single_ratio) {
  int pi, bh, tile, split, pidx;
  bool pair;
  unit_coords(P, P.nsplit, idx, pi, bh, tile, pair, split, pidx);
  const int b = bh / P.h;
  const int L = P.padding ? P.valid_len[b] : P.n_k;
  const int q_end = P.pad_queries ? (L < P.n_q ? L : P.n_q) : P.n_q;
  const int q0 = pi * 2 * BLK_M + tile * BLK_M;
  auto blocks = [&](int tq0) {
    if (tq0 >= q_end) return 0;
    int k_end = L;
    if (P.causal && tq0 + BLK_M < k_end) k_end = tq0 + BLK_M;
    int kb0;
    return split_range(P, P.nsplit, (k_end + BLK_N - 1) / BLK_N, split, kb0);
  };
  const double fixed = P.nsplit > 1 ? SPLIT_FIXED : 0.0;
  if (!pair) return blocks(q0) * single_ratio;
  return blocks(q0) + (q0 + BLK_M < P.n_q ? blocks(q0 + BLK_M) : 0) + fixed;
}

// Time of the static schedule of unit_index() on G persistent CTAs.
double persistent_makespan(const AttnTcParams& P, int G, double sr) {
  double worst = 0;
  for (int c = 0; c < G; ++c) {
    double t = 0;
    for (int i = 0;; ++i) {
      const int idx = unit_index_of(P, G, c, i);
      if (idx < 0) break;
      t += unit_cost_host(P, idx, sr) + PERSIST_FIXED;
    }
    worst = t > worst ? t : worst;
  }
  return worst;
}

// Time of one CTA per unit on G SMs: the hardware hands the units out in
// order, each to the first SM that becomes free.
double per_unit_makespan(const AttnTcParams& P, int G, double sr) {
  std::vector<double> free_at((size_t)G, 0.0);
  std::make_heap(free_at.begin(), free_at.end(), std::greater<double>());
  for (int idx = 0; idx < P.units; ++idx) {
    std::pop_heap(free_at.begin(), free_at.end(), std::greater<double>());
    free_at.back() += unit_cost_host(P, idx, sr) + UNIT_FIXED;
    std::push_heap(free_at.begin(), free_at.end(), std::greater<double>());
  }
  return *std::max_element(free_at.begin(), free_at.end());
}

// Key blocks of n_k keys.
int key_blocks(int n_k) { return (n_k + BLK_N - 1) / BLK_N; }

// Sets the split over the keys: at most `want` ranges of equal whole blocks
// (fewer when the blocks do not divide), every unit a tile pair.
void set_split(AttnTcParams& P, int want) {
  const int nb = key_blocks(P.n_k);
  if (want > nb) want = nb;
  if (want < 2) {
    P.nsplit = 1;
    P.split_blocks = nb;
    return;
  }
  P.split_blocks = (nb + want - 1) / want;
  P.nsplit = (nb + P.split_blocks - 1) / P.split_blocks;
  if (P.nsplit < 2) P.nsplit = 1;
  P.pi_major = 0;
  P.pair_units = P.units = P.npair * P.nbh * P.nsplit;
}

// Picks one CTA per unit or a persistent grid (and the unit order) for the
// shorter estimated time on G SMs; returns the grid size. max_split: the
// largest split over the keys allowed (1: none); a split is considered when
// the tile pairs alone leave SMs idle, and taken when its estimate is shorter.
int choose_schedule(AttnTcParams& P, int B, int d_h, int d_vh, int G, int max_split) {
  const int pairs = P.npair * P.nbh;
  const double sr = 1.0 + 4.0 * (d_h + d_vh) / 1600.0;
  P.pi_major = 0;
  P.nsplit = 1;
  P.split_blocks = key_blocks(P.n_k);
  P.pair_units = P.units = pairs;
  if (pairs <= G) {
    if (max_split < 2 || 2 * pairs > G) return pairs;
    // a split over the keys: s ranges per pair, all units in one round
    const double base = per_unit_makespan(P, G, sr);
    double best = base;
    int best_s = 1;
    for (int s = 2; s <= max_split && (long long)s * pairs <= G; ++s) {
      AttnTcParams S = P;
      set_split(S, s);
      if (S.nsplit < 2) break;
      const double t = per_unit_makespan(S, G, sr);
      if (t < best) {
        best = t;
        best_s = S.nsplit;
      }
    }
    if (best_s > 1) set_split(P, best_s);
    return P.units;
  }
  if (!P.causal && !P.padding) {
    // equal pairs: a persistent grid; the r pairs of a last, partly filled
    // round become 2 r single tiles when that shortens it
    const int r = pairs % G;
    if (r > 0 && 2 * r <= G && pairs <= MAX_SIMULATED_UNITS) {
      AttnTcParams S = P;
      S.pair_units = pairs - r;
      S.units = pairs + r;
      if (persistent_makespan(S, G, sr) < persistent_makespan(P, G, sr)) {
        P.pair_units = S.pair_units;
        P.units = S.units;
      }
    }
    return G;
  }
  if (pairs > MAX_SIMULATED_UNITS) return pairs;
  // the four schedules: one CTA per unit or persistent CTAs, units pair by
  // pair within each head or heavy causal pairs of all heads first (only
  // when the K and V that will be read stay in L2)
  double kv_bytes = 0;
  for (int b = 0; b < B; ++b)
    kv_bytes += (double)(P.padding ? P.valid_len[b] : P.n_k) * P.h * (d_h + d_vh) * 2.0;
  const bool pm_ok = P.causal && kv_bytes <= PI_MAJOR_MAX_KV_BYTES;
  double best = 0;
  int best_grid = pairs, best_pm = 0;
  for (int pm = 0; pm <= (pm_ok ? 1 : 0); ++pm) {
    P.pi_major = pm;
    const double one_each = per_unit_makespan(P, G, sr);
    const double persistent = persistent_makespan(P, G, sr);
    const double t = persistent < one_each ? persistent : one_each;
    if (pm == 0 || t < best) {
      best = t;
      best_grid = persistent < one_each ? G : pairs;
      best_pm = pm;
    }
  }
  P.pi_major = best_pm;
  return best_grid;
}

// A split over the keys fixed by the caller: nsplit ranges (at most one per
// key block), one CTA per unit, or a persistent grid when there are more
// units than SMs.
int forced_split_schedule(AttnTcParams& P, int nsplit, int G) {
  P.pi_major = 0;
  P.nsplit = 1;
  P.split_blocks = key_blocks(P.n_k);
  P.pair_units = P.units = P.npair * P.nbh;
  set_split(P, nsplit);
  return P.units <= G ? P.units : G;
}

template <int DQK, int DV, bool SPLIT>
mha_status launch_k(const AttnTcParams& P, int grid, cudaStream_t s) {
  using C = ACfg<DQK, DV>;
  if (!ensure_smem_limit((const void*)attn_tc_kernel<DQK, DV, SPLIT>, C::SMEM))
    return MHA_ERR_CUDA;
  const cudaError_t e = launch_dependent(attn_tc_kernel<DQK, DV, SPLIT>, dim3(grid),
                                         dim3(NTHREADS), C::SMEM, s, P);
  count_launch();
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

template <int DQK, bool SPLIT>
mha_status launch_sp_k(const AttnTcParams& P, int grid, cudaStream_t s) {
  using C = SpCfg<DQK>;
  if (!ensure_smem_limit((const void*)attn_tc_sp_kernel<DQK, SPLIT>, C::SMEM))
    return MHA_ERR_CUDA;
  const cudaError_t e = launch_dependent(attn_tc_sp_kernel<DQK, SPLIT>, dim3(grid),
                                         dim3(SP_THREADS), C::SMEM, s, P);
  count_launch();
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

// The kernels are compiled with and without the split's code, so that a
// launch without a split runs exactly the unsplit kernel.
template <int DQK, int DV>
mha_status launch(const AttnTcParams& P, int grid, cudaStream_t s) {
  return P.nsplit > 1 ? launch_k<DQK, DV, true>(P, grid, s) : launch_k<DQK, DV, false>(P, grid, s);
}

template <int DQK>
mha_status launch_sp(const AttnTcParams& P, int grid, cudaStream_t s) {
  return P.nsplit > 1 ? launch_sp_k<DQK, true>(P, grid, s) : launch_sp_k<DQK, false>(P, grid, s);
}



// The units of an attention call: tile pairs of every (batch item, head),
// with the lengths the masks use. Host only, no device work.
mha_status set_units(AttnTcParams& P, const AttnArgs& a) {
  P.n_q = a.n_q;
  P.n_k = a.n_k;
  P.h = a.h;
  P.npair = (a.n_q + 2 * BLK_M - 1) / (2 * BLK_M);
  const long long units = (long long)P.npair * a.h * a.B;
  if (units > (1ll << 29)) return MHA_ERR_UNSUPPORTED;
  P.units = P.pair_units = (int)units;
  P.nbh = a.h * a.B;
  P.causal = a.causal;
  P.padding = a.padding;
  P.pad_queries = a.pad_queries;
  for (int b = 0; b < MHA_MAX_PADDED_BATCH; ++b)
    P.valid_len[b] = (a.padding && b < a.B) ? a.valid_len_host[b] : a.n_k;
  return MHA_OK;
}

int split_dv(int d_vh) { return d_vh <= 64 ? 64 : 128; }

size_t split_counter_bytes(int pairs) {
  return ((size_t)pairs * 2 * sizeof(int) + 255) / 256 * 256;
}

// Largest split the automatic choice considers: all units in one round of at
// most SPLIT_SM_BOUND SMs (GB300 has 152), at most MAX_SPLITS ranges and one
// key block per range.
constexpr int SPLIT_SM_BOUND = 160;
constexpr int MAX_SPLITS = 64;

int auto_cap(int pairs, int n_k) {
  if (2 * (long long)pairs > SPLIT_SM_BOUND) return 1;
  int cap = SPLIT_SM_BOUND / pairs;
  if (cap > MAX_SPLITS) cap = MAX_SPLITS;
  if (cap > key_blocks(n_k)) cap = key_blocks(n_k);
  return cap < 1 ? 1 : cap;
}

// Resolves the split request of a call: sets the schedule in P and returns
// the grid, or -1 when a requested split does not fit the scratch.
int plan_call(AttnTcParams& P, const AttnArgs& a, int G) {
  const int pairs = P.npair * P.nbh;
  if (a.nsplit > 1) {
    const int grid = forced_split_schedule(P, a.nsplit, G);
    if (P.nsplit > 1 &&
        (!a.split_ws || a.split_ws_bytes < attention_split_bytes(a.B, a.n_q, a.h, a.d_vh, P.nsplit)))
      return -1;
    return grid;
  }
  int max_split = 1;
  if (a.nsplit == 0 && a.split_ws) {
    max_split = auto_cap(pairs, a.n_k);
    while (max_split > 1 &&
           attention_split_bytes(a.B, a.n_q, a.h, a.d_vh, max_split) > a.split_ws_bytes)
      --max_split;
  }
  return choose_schedule(P, a.B, a.d_h, a.d_vh, G, max_split);
}

// The schedule of the last few (shape, lengths, SM count, split request)
// seen, so that repeated calls skip the host simulation (up to ~0.2 ms per
// call on a large causal problem). Any schedule plan_call returns for a
// shape covers every (query tile, key block) whatever the lengths, so a hash
// collision of the lengths could only cost speed, never correctness.
struct PlanKey {
  int B, n_q, n_k, h, d_h, d_vh, causal, padding, pad_queries, G, nsplit, has_ws;
  size_t ws_bytes;
  uint64_t lens_hash;
  bool operator==(const PlanKey& o) const {
    return B == o.B && n_q == o.n_q && n_k == o.n_k && h == o.h && d_h == o.d_h &&
           d_vh == o.d_vh && causal == o.causal && padding == o.padding &&
           pad_queries == o.pad_queries && G == o.G && nsplit == o.nsplit &&
           has_ws == o.has_ws && ws_bytes == o.ws_bytes && lens_hash == o.lens_hash;
  }
};

struct PlanVal {
  int grid, units, pair_units, pi_major, nsplit, split_blocks;
};

int cached_plan(AttnTcParams& P, const AttnArgs& a, int G) {
  PlanKey k{a.B, a.n_q, a.n_k, a.h, a.d_h, a.d_vh, a.causal, a.padding, a.pad_queries, G,
            a.nsplit, a.split_ws != nullptr, a.split_ws_bytes, 1469598103934665603ull};
  if (a.padding)
    for (int b = 0; b < a.B; ++b)  // FNV-1a over the lengths
      k.lens_hash = (k.lens_hash ^ (uint32_t)a.valid_len_host[b]) * 1099511628211ull;
  constexpr int N = 16;
  static std::mutex mu;
  static PlanKey keys[N];
  static PlanVal vals[N];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (keys[i] == k) {
        const PlanVal& v = vals[i];
        P.units = v.units;
        P.pair_units = v.pair_units;
        P.pi_major = v.pi_major;
        P.nsplit = v.nsplit;
        P.split_blocks = v.split_blocks;
        return v.grid;
      }
  }
  const int grid = plan_call(P, a, G);
  if (grid < 0) return grid;
  std::lock_guard<std::mutex> lock(mu);
  keys[next] = k;
  vals[next] = PlanVal{grid, P.units, P.pair_units, P.pi_major, P.nsplit, P.split_blocks};
  next = (next + 1) % N;
  if (used < N) ++used;
  return grid;
}

}  // namespace

size_t attention_split_bytes(int B, int n_q, int h, int d_vh, int nsplit) {
  if (nsplit < 2) return 0;
  const long long pairs = (long long)((n_q + 2 * BLK_M - 1) / (2 * BLK_M)) * h * B;
  const int dv = split_dv(d_vh);
  return split_counter_bytes((int)pairs) +
         (size_t)pairs * 2 * nsplit * (size_t)(dv + 2) * BLK_M * sizeof(float);
}

size_t attention_split_counter_bytes(int B, int n_q, int h) {
  return split_counter_bytes((n_q + 2 * BLK_M - 1) / (2 * BLK_M) * h * B);
}

int attention_effective_splits(int n_k, int nsplit) {
  const int nb = key_blocks(n_k);
  if (nsplit > nb) nsplit = nb;
  if (nsplit < 2) return 1;
  const int per = (nb + nsplit - 1) / nsplit;
  const int n = (nb + per - 1) / per;
  return n < 2 ? 1 : n;
}

size_t attention_auto_split_bytes(int B, int n_q, int n_k, int h, int d_vh) {
  const long long pairs = (long long)((n_q + 2 * BLK_M - 1) / (2 * BLK_M)) * h * B;
  if (2 * pairs > SPLIT_SM_BOUND) return 0;
  return attention_split_bytes(B, n_q, h, d_vh, auto_cap((int)pairs, n_k));
}

mha_status attention_tc_plan(const AttnArgs& a, int num_sms, int* grid, int32_t* records,
                             size_t max_records, size_t* n_records) {
  AttnTcParams P;
  memset(&P, 0, sizeof(P));
  const mha_status st = set_units(P, a);
  if (st != MHA_OK) return st;
  const int G = plan_call(P, a, num_sms);
  if (G < 0) return MHA_ERR_WORKSPACE;
  *grid = G;
  size_t n = 0;
  for (int c = 0; c < G; ++c)
    for (int i = 0;; ++i) {
      const int idx = unit_index_of(P, G, c, i);
      if (idx < 0) break;
      if (records && n < max_records) {
        int pi, bh, tile, split, pidx;
        bool pair;
        unit_coords(P, P.nsplit, idx, pi, bh, tile, pair, split, pidx);
        int kb0;
        const int nkb = split_range(P, P.nsplit, key_blocks(P.n_k), split, kb0);
        int32_t* r = records + 7 * n;
        r[0] = c;
        r[1] = bh / P.h;
        r[2] = bh % P.h;
        r[3] = pi * 2 * BLK_M + tile * BLK_M;
        r[4] = pair ? 2 : 1;
        r[5] = kb0 * BLK_N;
        r[6] = std::min((kb0 + nkb) * BLK_N, P.n_k);
      }
      ++n;
    }
  *n_records = n;
  return MHA_OK;
}

mha_status attention_tc(const AttnArgs& a, cudaStream_t s) {
  AttnTcParams P;
  memset(&P, 0, sizeof(P));
  const uint64_t BH = (uint64_t)a.B * a.h;
  const uint64_t qd[3] = {(uint64_t)a.d_h, (uint64_t)a.n_q, BH};
  const uint64_t qs[2] = {(uint64_t)a.d_h * 2, (uint64_t)a.n_q * a.d_h * 2};
  const uint64_t kd[3] = {(uint64_t)a.d_h, (uint64_t)a.n_k, BH};
  const uint64_t ks[2] = {(uint64_t)a.d_h * 2, (uint64_t)a.n_k * a.d_h * 2};
  const uint64_t vd[3] = {(uint64_t)a.d_vh, (uint64_t)a.n_k, BH};
  const uint64_t vs[2] = {(uint64_t)a.d_vh * 2, (uint64_t)a.n_k * a.d_vh * 2};
  const uint32_t box[3] = {64, 128, 1};
  if (!make_tmap_bf16(&P.qmap, a.Q, 3, qd, qs, box, true) ||
      !make_tmap_bf16(&P.kmap, a.K, 3, kd, ks, box, true) ||
      !make_tmap_bf16(&P.vmap, a.V, 3, vd, vs, box, true))
    return MHA_ERR_CUDA;
  P.Z = a.Z;
  P.dv = a.d_vh;
  const mha_status st = set_units(P, a);
  if (st != MHA_OK) return st;
  // |c| log2(e), kept at 1e-30 or above so that a masked score (-inf) stays
  // -inf after scaling; for c = 0 (or |c| below that) every allowed score
  // scales to within 1e-26 of 0 and gets weight 2^0 = 1: the uniform
  // distribution over the allowed keys, as softmax of all-zero scores
  P.cl2 = fmaxf(fabsf(a.c) * 1.4426950408889634f, 1e-30f);
  P.negate = a.c < 0.f;
  P.err = a.err;
  P.limit_ns = wait_limit_ns();
  // a gate is only ever passed for h <= MHA_MAX_GATED_HEADS (checked by the
  // caller); without one every head is read with scale 1, for any h
  P.has_gate = a.head_gate_host != nullptr && a.h <= MHA_MAX_GATED_HEADS;
  for (int i = 0; i < MHA_MAX_GATED_HEADS; ++i)
    P.head_gate[i] = (P.has_gate && i < a.h) ? a.head_gate_host[i] : 1.f;
  // one CTA per unit, or one persistent CTA per SM walking its share; a
  // split over the keys when asked for, or when the tile pairs leave SMs idle
  const int grid = cached_plan(P, a, num_sms());
  if (grid < 0) return MHA_ERR_WORKSPACE;
  if (P.nsplit > 1) {
    const size_t cnt_bytes = split_counter_bytes(P.npair * P.nbh);
    P.split_cnt = static_cast<int*>(a.split_ws);
    P.part = reinterpret_cast<float*>(static_cast<char*>(a.split_ws) + cnt_bytes);
    if (!a.split_cnt_zeroed && cudaMemsetAsync(P.split_cnt, 0, cnt_bytes, s) != cudaSuccess)
      return MHA_ERR_CUDA;
  }
  // Head sizes of 32..64 run as 64 and those of 72..128 as 128: the columns
  // past d_h (past d_vh) of the 64-wide panels are read as zeros (TMA fill
  // past the tensor's extent), so the padded dot products are exact and z's
  // extra columns stay 0 and are not written. d_vh <= 64: S, P and z fit in
  // separate TMEM columns.
  if (a.d_h < 32 || a.d_h > 128 || a.d_vh < 32 || a.d_vh > 128) return MHA_ERR_UNSUPPORTED;
  const bool q64 = a.d_h <= 64, v64 = a.d_vh <= 64;
  if (q64 && v64) return launch_sp<64>(P, grid, s);
  if (!q64 && !v64) return launch<128, 128>(P, grid, s);
  if (q64) return launch<64, 128>(P, grid, s);
  return launch_sp<128>(P, grid, s);
}

}  // namespace mha
