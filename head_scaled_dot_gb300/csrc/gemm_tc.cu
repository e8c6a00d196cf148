// gemm_tc.cu - bf16 GEMM on tcgen05 tensor cores for the two projections:
//   QKV: Q = X_q W_Q, K = X_kv W_K, V = X_kv W_V with the head split
//        (B,T,h d) -> (B,h,T,d) done in the epilogue ("Multi-Head Attention
//        review", "Separate and Combined Projections");
//   out: Y = Z W_O ("The Complete Multi-Head Operation").
//
// Persistent kernel, one CTA per SM (or clusters of two, see gemm_tc_kernel),
// 128 x BN output tiles (BN = 256 or 128),
// 64-deep K blocks in a STAGES-deep shared-memory ring filled by TMA. The
// problems that share their A operand (the QKV projections of one input) form
// a group whose tiles run M panel by M panel, each 128-row panel of A through
// every problem of the group back to back, so each panel is read from memory
// once and then from L2. Panels that hold only padding rows are not
// multiplied (skipped, or for the output projection written as zeros).
//
//   warp 0      TMA producer (one thread)
//   warp 1      MMA issuer (one thread), owns the TMEM allocation
//   warps 2..5  epilogue: TMEM -> registers -> bf16 -> global
// The fp32 accumulator lives in TMEM, double-buffered (2 x BN columns) so the
// epilogue of one tile overlaps the main loop of the next. A is K-major
// (row-major X), B is MN-major (row-major W): both straight from the caller's
// layout, no transpose or packing pass.
#include <cuda_bf16.h>

#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace mha {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int MAXP = 3;
constexpr int MAXRUNS = MHA_MAX_PADDED_BATCH + 1;

// Launch parameters of the kernel; the run tables are sized by the template
// argument so that launches with few runs (no selection, or a few batch
// items) pass a small parameter block.
struct GemmTcHead {
  CUtensorMap amap[MAXP];  // A: dims {K, M}, box {64, 128}, 128B swizzle
  CUtensorMap bmap[MAXP];  // W: dims {N, K}, box {64, 64}, 128B swizzle
  GemmProblem prob[MAXP];
  int tiles_n[MAXP];       // N tiles of each problem
  int ngroups;
  int g_first[MAXP + 1];   // problems [g_first[g], g_first[g + 1]) form group g
  int g_ntiles[MAXP];      // N tiles of one M panel through all of group g
  int g_select[MAXP];      // group g multiplies only the selected panels
  int g_panels[MAXP];      // M panels of group g (selected ones only, for g_select)
  int g_start[MAXP + 1];   // first tile of group g; g_start[ngroups]: product tiles
  int zero_prob;           // problem whose unselected panels are written as zeros
  int zero_tiles;          // tiles [g_start[ngroups], + zero_tiles): zero fills
  int nrun, nzrun;
  int32_t* err;
  uint64_t limit_ns;
};

template <int RUNS>
struct GemmTcParams {
  GemmTcHead h;
  int run_m[RUNS];    // selected panels: run r starts at panel run_m[r]
  int run_pre[RUNS];  //   and is preceded by run_pre[r] selected panels
  int zrun_m[RUNS];   // unselected panels, the same way
  int zrun_pre[RUNS];
};

constexpr int SMALL_RUNS = 8;

// CL = 1: one CTA, a 128 x BN tile, A and the whole W tile in its shared
// memory. CL = 2: a CTA pair computes a 256 x BN tile with cta_group::2
// MMAs; each CTA holds its 128 rows of A and half of the W tile, so a stage
// is smaller and the ring deeper in the same shared memory.
template <int BN, int CL>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;         // 16 KB
  static constexpr int B_BYTES = BK * (BN / CL) * 2;  // this CTA's part of the W tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // epilogue staging: per epilogue warp 32 rows x 64 columns of bf16
  static constexpr int STAGING_BYTES = 4 * 32 * 128;
  static constexpr int BUDGET = 227 * 1024 - STAGING_BYTES - 1024 /*align*/ - 256 /*barriers*/;
  static constexpr int STAGES = BUDGET / STAGE_BYTES > 8 ? 8 : BUDGET / STAGE_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // double-buffered accumulator
  static_assert(STAGES >= 4, "shared memory");
};

// The k-th panel of a run table (runs sorted, k below the table's total).
__device__ __forceinline__ int panel_of(const int* run_m, const int* run_pre, int nrun, int k) {
  int lo = 0, hi = nrun - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (run_pre[mid] <= k)
      lo = mid;
    else
      hi = mid - 1;
  }
  return run_m[lo] + (k - run_pre[lo]);
}

struct Tile {
  int p, m0, n0;
  bool zero;  // write zeros, no product
};

// Product tile t of a cluster of CL CTAs, for the CTA of rank `rank`: the
// cluster's tiles have the same N tile and CL consecutive M panels of one
// group (a panel past the group's last is a tile of rows past M: its A loads
// are zero fill and its rows are not stored).
template <class Params>
__device__ __forceinline__ Tile decode_tile(const Params& P, int t, int bn, int CL, int rank) {
  const GemmTcHead& H = P.h;
  Tile r;
  int g = 0;
  while (g + 1 < H.ngroups && t >= H.g_start[g + 1]) ++g;
  const int local = t - H.g_start[g];
  const int k = local / H.g_ntiles[g];
  int rr = local % H.g_ntiles[g];
  int p = H.g_first[g];
  while (rr >= H.tiles_n[p]) rr -= H.tiles_n[p++];
  r.p = p;
  const int panel = CL * k + rank;
  if (panel >= H.g_panels[g])
    r.m0 = (H.prob[p].M + BM - 1) / BM * BM;
  else
    r.m0 = (H.g_select[g] ? panel_of(P.run_m, P.run_pre, H.nrun, panel) : panel) * BM;
  r.n0 = rr * bn;
  r.zero = false;
  return r;
}

// Zero-fill tile z (rows with nothing to multiply).
template <class Params>
__device__ __forceinline__ Tile decode_zero_tile(const Params& P, int z, int bn) {
  const GemmTcHead& H = P.h;
  Tile r;
  const int tn = H.tiles_n[H.zero_prob];
  r.p = H.zero_prob;
  r.m0 = panel_of(P.zrun_m, P.zrun_pre, H.nzrun, z / tn) * BM;
  r.n0 = (z % tn) * bn;
  r.zero = true;
  return r;
}

// A bounded wait that ignores the abort flag: used only while draining
// operations this CTA itself started, before it releases shared memory/TMEM.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if (globaltimer_ns() - t0 > 100000000ull) return;  // 100 ms
  }
}

// Output offset of row m's element (m, n) through the problem's index map,
// split into the row part (row_offset) and the column part.
__device__ __forceinline__ long long row_offset(const GemmProblem& pr, int m) {
  return (long long)(m / pr.rows_per_group) * pr.s_group_row +
         (long long)(m % pr.rows_per_group) * pr.s_row;
}

// Writes a warp's 32 rows x 64 columns [n, n + 64) of a tile (rows m0w ..
// m0w + 31) to the output: the rows sit in the warp's shared-memory staging
// area `st` (row r: 8 chunks of 8 bf16, chunk k at position k ^ (r & 7)),
// and each store instruction writes 4 rows x 128 contiguous bytes. `rowoff`
// is lane r's row_offset of row m0w + r (valid when that row is below M);
// `zero`: write zeros instead of the staged values. Every 8-column chunk
// lies inside one column group (N and cols_per_group are multiples of 8), so
// it is stored whole or, past N, not at all.
__device__ __forceinline__ void store_warp_rows(const GemmProblem& pr, const uint4* st, int m0w,
                                                long long rowoff, int n, bool zero, int lane) {
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(pr.out);
  // a lane always stores chunk cc = lane % 8 of rows 4 it + lane / 8
  const int cc = lane & 7;
  const int nn = n + 8 * cc;
  const long long coloff =
      (long long)(nn / pr.cols_per_group) * pr.s_group_col + (nn % pr.cols_per_group);
  const bool col_ok = nn < pr.N;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = 4 * it + (lane >> 3);
    const long long ro = __shfl_sync(0xffffffffu, rowoff, r);
    if (col_ok && m0w + r < pr.M) {
      const uint4 v = zero ? make_uint4(0, 0, 0, 0) : st[r * 8 + (cc ^ (r & 7))];
      *reinterpret_cast<uint4*>(out + ro + coloff) = v;
    }
  }
}

// CL = 2: the kernel runs in clusters of two CTAs that compute a 256 x BN
// tile (two vertically adjacent M panels, the same N tile) with cta_group::2
// MMAs issued by one thread of the even CTA. Each CTA loads its own A panel
// and its half of the W tile into its own shared memory (the W tile is read
// from L2 once per pair, and a stage is 32 KB instead of 48 KB, so the ring
// is six stages deep instead of four); the bytes of both CTAs complete on the
// even CTA's full barrier, the issuer's commits arrive on both CTAs' empty
// and accumulator barriers, and each CTA's epilogue reads its 128 rows of the
// accumulator from its own tensor memory and frees it on the issuer's
// barrier.
template <int BN, int RUNS, int CL>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ GemmTcParams<RUNS> P) {
  using C = Cfg<BN, CL>;
  const GemmTcHead& H = P.h;
  const int rank = CL > 1 ? (int)cluster_rank() : 0;
  const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;  // cluster and clusters
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint4* staging = reinterpret_cast<uint4*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::STAGING_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);   // the (even CTA's) producer; the bytes of both CTAs
      mbar_init(&empty[s], 1);  // one MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4 * CL);  // one arrival per epilogue warp of the pair
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // The producer thread fetches the descriptors and decodes its first tile
  // (parameters only) before the grid dependency wait, so that its first
  // loads go out as soon as the previous kernel's results may be read.
  const int prod = H.g_start[H.ngroups];  // product tiles (per cluster)
  Tile first{};
  if (threadIdx.x == 0) {
    for (int p = 0; p < MAXP; ++p) {
      if (p >= H.g_first[H.ngroups]) break;
      tma_prefetch_desc(&H.amap[p]);
      tma_prefetch_desc(&H.bmap[p]);
    }
    if (cid < prod) first = decode_tile(P, cid, BN, CL, rank);
  }
  if (warp == 1) {
    if (CL == 1) {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    }
  }
  tc_fence_before();
  __syncthreads();
  // the other CTA's barriers are initialized before either signals them
  if (CL > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The prologue above touched only this CTA's shared and tensor memory. The
  // next kernel may start its own now; this one reads its inputs and writes
  // its outputs only once the previous kernel has completed.
  grid_dep_launch_dependents();
  grid_dep_wait();
  const WaitCtl w{H.err, abort_flag, H.limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;  // global k-block counter across tiles
      bool ok = true;
      for (int t = cid; t < prod && ok; t += ncl) {
        const Tile tl = t == cid ? first : decode_tile(P, t, BN, CL, rank);
        const int kblocks = (H.prob[tl.p].K + BK - 1) / BK;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (it >= (uint32_t)C::STAGES && !mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1, w)) {
            ok = false;
            break;
          }
          uint8_t* a_s = smem + s * C::STAGE_BYTES;
          uint8_t* b_s = a_s + C::A_BYTES;
          if (CL == 1) {
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
            tma_load_2d(a_s, &H.amap[tl.p], &full[s], kb * BK, tl.m0);
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(b_s + j * (BK * 128), &H.bmap[tl.p], &full[s], tl.n0 + 64 * j, kb * BK);
          } else {
            // this CTA's A panel and its half of the W tile, into its own
            // shared memory; the bytes of both CTAs complete on the even
            // CTA's full barrier, which expects them all
            if (rank == 0) mbar_arrive_expect_tx(&full[s], CL * C::STAGE_BYTES);
            const uint32_t fb = cluster_addr(&full[s], 0);
            tma_load_2d_pair(a_s, &H.amap[tl.p], fb, kb * BK, tl.m0);
            constexpr int PER = BN / 64 / CL;
#pragma unroll
            for (int j = 0; j < PER; ++j)
              tma_load_2d_pair(b_s + j * (BK * 128), &H.bmap[tl.p], fb,
                               tl.n0 + 64 * (rank * PER + j), kb * BK);
          }
        }
      }
      if (!ok && rank == 0) {  // let the loads of this stage ring land before it exits
        for (uint32_t k = (it > (uint32_t)C::STAGES ? it - C::STAGES : 0); k < it; ++k)
          drain_wait(&full[k % C::STAGES], (k / C::STAGES) & 1);
      }
      if (CL > 1) {
        // the even CTA's last commits arrive on this CTA's empty barriers:
        // they must have landed before this CTA's shared memory is released
        for (uint32_t k = (it > (uint32_t)C::STAGES ? it - C::STAGES : 0); k < it; ++k)
          drain_wait(&empty[k % C::STAGES], (k / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // the MMA issuer: every CTA (CL = 1) or the even CTA of a pair
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM * CL, BN, 0, 1);
      uint32_t it = 0, tile_i = 0;
      bool ok = true;
      for (int t = cid; t < prod && ok; t += ncl, ++tile_i) {
        const Tile tl = decode_tile(P, t, BN, CL, rank);
        const int kblocks = (H.prob[tl.p].K + BK - 1) / BK;
        const uint32_t buf = tile_i & 1;
        // wait until the epilogue has drained this accumulator buffer
        if (tile_i >= 2 && !mbar_wait(&acc_empty[buf], ((tile_i >> 1) - 1) & 1, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (!mbar_wait(&full[s], (it / C::STAGES) & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A K-major: advance 16 elements (32 B) inside the 128 B swizzle row.
            const uint64_t ad = sdesc_sw128(a_addr + kk * 32, 16, 1024);
            // B MN-major: 16 K-rows of 128 B each; 64-column panels 8 KB apart.
            const uint64_t bd = sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024);
            if (CL == 1)
              umma_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0);
            else
              umma_ss_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
          }
          // frees the stage (in both CTAs of a pair) once these MMAs finish
          if (CL == 1)
            umma_commit(&empty[s]);
          else
            umma_commit_pair_mc(&empty[s], 3);
        }
        if (ok) {
          if (CL == 1)
            umma_commit(&acc_full[buf]);
          else
            umma_commit_pair_mc(&acc_full[buf], 3);
        }
      }
      if (!ok) {  // wait for this thread's MMAs before TMEM is released
        uint64_t* last = &acc_full[0];
        if (CL == 1)
          umma_commit(last);
        else
          umma_commit_pair_mc(last, 1);
        drain_wait(last, 0);
        drain_wait(last, 1);
      }
    }
  } else {
    // Epilogue warps 2..5: warp w reads TMEM lanes 32*(w%4) .. +31. First
    // this CTA's zero fills (one CTA at a time over the zero tiles), while
    // the first product tile is still being multiplied; then the cluster's
    // product tiles. Rows go out through the warp's staging area, 4 rows of
    // 128 contiguous bytes per store instruction.
    const int g = warp & 3;
    uint4* st = staging + g * (32 * 8);
    for (int z = blockIdx.x; z < H.zero_tiles; z += (int)gridDim.x) {
      const Tile tl = decode_zero_tile(P, z, BN);
      const GemmProblem& pr = H.prob[tl.p];
      const int m0w = tl.m0 + 32 * g;
      const long long ro = m0w + lane < pr.M ? row_offset(pr, m0w + lane) : 0;
      for (int c = 0; c < BN; c += 64) store_warp_rows(pr, st, m0w, ro, tl.n0 + c, true, lane);
    }
    uint32_t tile_i = 0;
    bool ok = true;
    const int nprod = (prod - cid + ncl - 1) / ncl;  // product tiles of this CTA
    for (int i = 0; i < nprod; ++i) {
      const Tile tl = decode_tile(P, cid + i * ncl, BN, CL, rank);
      const GemmProblem& pr = H.prob[tl.p];
      const int m0w = tl.m0 + 32 * g;
      const long long ro = m0w + lane < pr.M ? row_offset(pr, m0w + lane) : 0;
      const uint32_t buf = tile_i & 1;
      const uint32_t phase = (tile_i >> 1) & 1;
      ++tile_i;
      if (!ok || !mbar_wait(&acc_full[buf], phase, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + buf * BN + (static_cast<uint32_t>(32 * g) << 16);
#pragma unroll 1
      for (int c = 0; c < BN; c += 64) {
        uint32_t r0[32], r1[32];
        tmem_ld32(taddr + c, r0);
        tmem_ld32(taddr + c + 32, r1);
        tmem_wait_ld();
        // this lane's row, columns [c, c + 64): 8 chunks of 8 bf16
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t* src = k < 4 ? r0 + 8 * k : r1 + 8 * (k - 4);
          st[lane * 8 + (k ^ (lane & 7))] =
              make_uint4(pack_bf16x2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                         pack_bf16x2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                         pack_bf16x2(__uint_as_float(src[4]), __uint_as_float(src[5])),
                         pack_bf16x2(__uint_as_float(src[6]), __uint_as_float(src[7])));
        }
        __syncwarp();
        store_warp_rows(pr, st, m0w, ro, tl.n0 + c, false, lane);
        __syncwarp();  // the staging area is rewritten by the next chunk
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CL == 1)
          mbar_arrive(&acc_empty[buf]);
        else
          mbar_arrive_cluster(cluster_addr(&acc_empty[buf], 0));  // the issuer's barrier
      }
    }
  }
  // Every lane of a warp meets here before the CTA-wide barrier: a barrier
  // counts whole warps, so a warp must not reach it split across branches.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // neither CTA of a cluster leaves while the other may still write into it
  if (CL > 1) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (CL == 1)
      tmem_dealloc(tmem, C::TMEM_COLS);
    else
      tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

// Clusters of CL CTAs of this kernel that can be resident at once on the
// current device (a cluster's CTAs share a GPC), asked once per device.
template <int BN, int RUNS, int CL>
int max_clusters() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms() / CL;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * (num_sms() / CL));
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = Cfg<BN, CL>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, RUNS, CL>, &cfg) != cudaSuccess ||
        n < 1)
      n = num_sms() / CL;
    cached[dev] = n;
  }
  return cached[dev];
}

// Clusters of the paired kernel that fit at once (0 if its shared memory
// cannot be granted).
template <int BN>
int pair_clusters() {
  if (!ensure_smem_limit((const void*)gemm_tc_kernel<BN, SMALL_RUNS, 2>, Cfg<BN, 2>::SMEM)) return 0;
  return max_clusters<BN, SMALL_RUNS, 2>();
}

template <int BN, int RUNS, int CL>
mha_status launch_kernel(const GemmTcParams<RUNS>& P, int clusters, cudaStream_t s) {
  using C = Cfg<BN, CL>;
  auto kernel = gemm_tc_kernel<BN, RUNS, CL>;
  if (!ensure_smem_limit((const void*)kernel, C::SMEM)) return MHA_ERR_CUDA;
  const int cap = max_clusters<BN, RUNS, CL>();
  if (clusters > cap) clusters = cap;
  const int grid = clusters * CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, P);
  count_launch();
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

// Tiles per cluster of CL CTAs: a group's M panels are taken CL at a time.
template <int BN, int CL>
mha_status launch(GemmTcParams<MAXRUNS>& P, int nprob, int sel_panels, int unsel_panels,
                  cudaStream_t s) {
  GemmTcHead& H = P.h;
  for (int i = 0; i < nprob; ++i) H.tiles_n[i] = (H.prob[i].N + BN - 1) / BN;
  int start = 0;
  for (int g = 0; g < H.ngroups; ++g) {
    int nt = 0;
    for (int p = H.g_first[g]; p < H.g_first[g + 1]; ++p) nt += H.tiles_n[p];
    H.g_ntiles[g] = nt;
    const GemmProblem& pr = H.prob[H.g_first[g]];
    const long long panels = H.g_select[g] ? sel_panels : (pr.M + BM - 1) / BM;
    if (panels > (1ll << 30)) return MHA_ERR_UNSUPPORTED;
    H.g_panels[g] = (int)panels;
    H.g_start[g] = start;
    const long long tiles = (long long)start + (panels + CL - 1) / CL * nt;
    if (tiles > (1ll << 30)) return MHA_ERR_UNSUPPORTED;
    start = (int)tiles;
  }
  H.g_start[H.ngroups] = start;
  H.zero_tiles = H.zero_prob >= 0 ? unsel_panels * H.tiles_n[H.zero_prob] : 0;
  // clusters for the product tiles, and CTAs enough for the zero fills
  int clusters = start;
  const int zero_cl = (H.zero_tiles + CL - 1) / CL;
  if (zero_cl > clusters) clusters = zero_cl;
  if (clusters > num_sms() / CL) clusters = num_sms() / CL;
  if (clusters < 1) clusters = 1;
  if (H.nrun <= SMALL_RUNS && H.nzrun <= SMALL_RUNS) {
    GemmTcParams<SMALL_RUNS> Q;
    Q.h = H;
    for (int r = 0; r < SMALL_RUNS; ++r) {
      Q.run_m[r] = P.run_m[r];
      Q.run_pre[r] = P.run_pre[r];
      Q.zrun_m[r] = P.zrun_m[r];
      Q.zrun_pre[r] = P.zrun_pre[r];
    }
    return launch_kernel<BN, SMALL_RUNS, CL>(Q, clusters, s);
  }
  return launch_kernel<BN, MAXRUNS, CL>(P, clusters, s);
}

// Runs of selected and of unselected 128-row panels of the B * rows_per_batch
// rows: panel k is selected when it holds a row j < need[b] of some batch item
// b. Returns false when a table would overflow.
bool build_runs(const RowSelect& sel, GemmTcParams<MAXRUNS>& P, int& sel_panels,
                int& unsel_panels) {
  const long long T = sel.rows_per_batch;
  const long long panels = (sel.B * T + BM - 1) / BM;
  int n = 0, cnt = 0;
  long long last_end = -1;  // one past the last selected panel so far
  for (int b = 0; b < sel.B; ++b) {
    const long long first = b * T / BM, end = (b * T + sel.need[b] - 1) / BM + 1;
    if (n > 0 && first <= last_end) {  // overlaps or touches the current run
      if (end > last_end) {
        cnt += (int)(end - last_end);
        last_end = end;
      }
      continue;
    }
    if (n >= MAXRUNS) return false;
    P.run_m[n] = (int)first;
    P.run_pre[n] = cnt;
    ++n;
    cnt += (int)(end - first);
    last_end = end;
  }
  P.h.nrun = n;
  sel_panels = cnt;
  // the complement
  int z = 0, zc = 0;
  long long pos = 0;
  for (int r = 0; r <= n; ++r) {
    const long long gap_end = r < n ? P.run_m[r] : panels;
    const long long run_len = r < n ? (r + 1 < n ? P.run_pre[r + 1] : cnt) - P.run_pre[r] : 0;
    if (gap_end > pos) {
      if (z >= MAXRUNS) return false;
      P.zrun_m[z] = (int)pos;
      P.zrun_pre[z] = zc;
      ++z;
      zc += (int)(gap_end - pos);
    }
    pos = gap_end + run_len;
  }
  P.h.nzrun = z;
  unsel_panels = zc;
  return true;
}

}  // namespace

mha_status gemm_tc(const GemmProblem* probs, int nprob, const RowSelect* sel, int32_t* err,
                   cudaStream_t s) {
  if (nprob < 1 || nprob > MAXP) return MHA_ERR_INVALID_ARG;
  static thread_local GemmTcParams<MAXRUNS> P;  // 17 KB: off the stack
  memset(&P, 0, sizeof(P));
  GemmTcHead& H = P.h;
  H.err = err;
  H.limit_ns = wait_limit_ns();
  H.zero_prob = -1;
  bool all256 = true;
  int nsel = 0;
  for (int i = 0; i < nprob; ++i) {
    const GemmProblem& pr = probs[i];
    H.prob[i] = pr;
    if (pr.select) {
      if (!sel || sel->B < 1 || sel->B > MHA_MAX_PADDED_BATCH ||
          (long long)sel->B * sel->rows_per_batch != pr.M)
        return MHA_ERR_INVALID_ARG;
      ++nsel;
    }
    if (pr.N % 256) all256 = false;
    // A: row-major M x K (K contiguous).
    const uint64_t adims[2] = {(uint64_t)pr.K, (uint64_t)pr.M};
    const uint64_t astr[1] = {(uint64_t)pr.K * 2};
    const uint32_t abox[2] = {64, BM};
    // W: row-major K x N (N contiguous), loaded as 64-column panels.
    const uint64_t bdims[2] = {(uint64_t)pr.N, (uint64_t)pr.K};
    const uint64_t bstr[1] = {(uint64_t)pr.N * 2};
    const uint32_t bbox[2] = {64, BK};
    if (!make_tmap_bf16(&H.amap[i], pr.A, 2, adims, astr, abox, true) ||
        !make_tmap_bf16(&H.bmap[i], pr.W, 2, bdims, bstr, bbox, true))
      return MHA_ERR_CUDA;
    // 16-byte vector stores in the epilogue: every row pitch, group stride and
    // 32-column chunk offset is a multiple of 8 elements
    if (pr.cols_per_group % 8 || pr.N % 8 || pr.s_row % 8 || pr.s_group_col % 8 ||
        pr.s_group_row % 8)
      return MHA_ERR_UNSUPPORTED;
  }
  // groups: neighbours with the same A operand and the same row selection
  H.ngroups = 0;
  for (int i = 0; i < nprob; ++i) {
    const GemmProblem& pr = probs[i];
    const bool join = i > 0 && pr.A == probs[i - 1].A && pr.M == probs[i - 1].M &&
                      pr.K == probs[i - 1].K && pr.select == probs[i - 1].select;
    if (!join) {
      H.g_first[H.ngroups] = i;
      H.g_select[H.ngroups] = pr.select;
      ++H.ngroups;
    }
  }
  H.g_first[H.ngroups] = nprob;
  int sel_panels = 0, unsel_panels = 0;
  if (nsel > 0) {
    for (int b = 0; b < sel->B; ++b)
      if (sel->need[b] < 1 || sel->need[b] > sel->rows_per_batch) return MHA_ERR_INVALID_ARG;
    if (!build_runs(*sel, P, sel_panels, unsel_panels)) return MHA_ERR_UNSUPPORTED;
    if (sel->zero_rest) {
      if (nprob != 1) return MHA_ERR_INVALID_ARG;
      H.zero_prob = 0;
    }
  }
  // CTA pairs (256-row tiles, half of the W tile in each CTA's shared
  // memory, a deeper ring) when their rounds over the clusters that fit at
  // once are not more than the single CTAs' rounds over the SMs by the ~8 %
  // a paired tile is faster by (measured on GB300: 3-7 % on the grouped
  // projections; an output projection whose tiles fill whole rounds of
  // single CTAs but not of pairs was 6 % slower in pairs).
  const int bn = all256 ? 256 : 128;
  long long tiles = 0, pair_tiles = 0;
  for (int g = 0; g < H.ngroups; ++g) {
    long long nt = 0;
    for (int p = H.g_first[g]; p < H.g_first[g + 1]; ++p) nt += (probs[p].N + bn - 1) / bn;
    const GemmProblem& pr = probs[H.g_first[g]];
    const long long panels = H.g_select[g] ? sel_panels : (pr.M + BM - 1) / BM;
    tiles += panels * nt;
    pair_tiles += (panels + 1) / 2 * nt;
  }
  const int sms = num_sms();
  const int clusters = all256 ? pair_clusters<256>() : pair_clusters<128>();
  const long long rounds = (tiles + sms - 1) / sms;
  const long long pair_rounds = clusters > 0 ? (pair_tiles + clusters - 1) / clusters : rounds + 1;
  const bool pair = pair_rounds * 100 <= rounds * 108;
  if (!pair)
    return all256 ? launch<256, 1>(P, nprob, sel_panels, unsel_panels, s)
                  : launch<128, 1>(P, nprob, sel_panels, unsel_panels, s);
  return all256 ? launch<256, 2>(P, nprob, sel_panels, unsel_panels, s)
                : launch<128, 2>(P, nprob, sel_panels, unsel_panels, s);
}

}  // namespace mha
