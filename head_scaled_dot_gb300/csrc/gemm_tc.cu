// gemm_tc.cu - bf16 GEMM on tcgen05 tensor cores for the two projections:
//   QKV: Q = X_q W_Q, K = X_kv W_K, V = X_kv W_V with the head split
//        (B,T,h d) -> (B,h,T,d) done in the epilogue ("Multi-Head Attention
//        review", "Separate and Combined Projections");
//   out: Y = Z W_O ("The Complete Multi-Head Operation").
//
// Persistent kernel, one CTA per SM, 128 x BN output tiles (BN = 256 or 128),
// 64-deep K blocks in a STAGES-deep shared-memory ring filled by TMA:
//   warp 0      TMA producer (one thread)
//   warp 1      MMA issuer (one thread), owns the TMEM allocation
//   warps 2..5  epilogue: TMEM -> registers -> bf16 -> global
// The fp32 accumulator lives in TMEM, double-buffered (2 x BN columns) so the
// epilogue of one tile overlaps the main loop of the next. A is K-major
// (row-major X), B is MN-major (row-major W): both straight from the caller's
// layout, no transpose or packing pass.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "internal.h"

namespace mha {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int MAXP = 3;

struct GemmTcParams {
  CUtensorMap amap[MAXP];  // A: dims {K, M}, box {64, 128}, 128B swizzle
  CUtensorMap bmap[MAXP];  // W: dims {N, K}, box {64, 64}, 128B swizzle
  GemmProblem prob[MAXP];
  int tiles_n[MAXP];       // N tiles per problem
  int tile_start[MAXP + 1];
  int nprob;
  int32_t* err;
  uint64_t limit_ns;
};

template <int BN>
struct Cfg {
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr int A_BYTES = BM * BK * 2;   // 16 KB
  static constexpr int B_BYTES = BK * BN * 2;   // 32 KB (BN = 256)
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // double-buffered accumulator
};

__device__ __forceinline__ void decode_tile(const GemmTcParams& P, int t, int& p, int& m0,
                                            int& n0, int bn) {
  p = 0;
  while (p + 1 < P.nprob && t >= P.tile_start[p + 1]) ++p;
  const int local = t - P.tile_start[p];
  const int tn = P.tiles_n[p];
  m0 = (local / tn) * BM;
  n0 = (local % tn) * bn;
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

template <int BN>
__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ GemmTcParams P) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
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
  const int total = P.tile_start[P.nprob];

  if (warp == 0) {
    if (lane == 0) {
      for (int p = 0; p < P.nprob; ++p) {
        tma_prefetch_desc(&P.amap[p]);
        tma_prefetch_desc(&P.bmap[p]);
      }
      uint32_t it = 0;  // global k-block counter across tiles
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int p, m0, n0;
        decode_tile(P, t, p, m0, n0, BN);
        const int kblocks = (P.prob[p].K + BK - 1) / BK;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (it >= (uint32_t)C::STAGES && !mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1, w)) {
            ok = false;
            break;
          }
          uint8_t* a_s = smem + s * C::STAGE_BYTES;
          uint8_t* b_s = a_s + C::A_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(a_s, &P.amap[p], &full[s], kb * BK, m0);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(b_s + j * (BK * 128), &P.bmap[p], &full[s], n0 + 64 * j, kb * BK);
        }
      }
      if (!ok) {  // let the loads this CTA started land before it exits
        for (uint32_t k = (it > (uint32_t)C::STAGES ? it - C::STAGES : 0); k < it; ++k)
          drain_wait(&full[k % C::STAGES], (k / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 1);
      uint32_t it = 0, tile_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tile_i) {
        int p, m0, n0;
        decode_tile(P, t, p, m0, n0, BN);
        const int kblocks = (P.prob[p].K + BK - 1) / BK;
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
            umma_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0);
          }
          umma_commit(&empty[s]);  // frees the stage once these MMAs finish
        }
        if (ok) umma_commit(&acc_full[buf]);
      }
      if (!ok) {  // wait for this thread's MMAs before TMEM is released
        uint64_t* last = &acc_full[0];
        umma_commit(last);
        drain_wait(last, 0);
        drain_wait(last, 1);
      }
    }
  } else {
    // Epilogue warps 2..5: warp w reads TMEM lanes 32*(w%4) .. +31.
    const int g = warp & 3;
    uint32_t tile_i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tile_i) {
      int p, m0, n0;
      decode_tile(P, t, p, m0, n0, BN);
      const uint32_t buf = tile_i & 1;
      if (!mbar_wait(&acc_full[buf], (tile_i >> 1) & 1, w)) break;
      tc_fence_after();
      const GemmProblem& pr = P.prob[p];
      const int m = m0 + 32 * g + lane;
      const bool row_ok = m < pr.M;
      long long row_off = 0;
      if (row_ok)
        row_off = (long long)(m / pr.rows_per_group) * pr.s_group_row +
                  (long long)(m % pr.rows_per_group) * pr.s_row;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(pr.out);
      const uint32_t taddr = tmem + buf * BN + (static_cast<uint32_t>(32 * g) << 16);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c, r);
        tmem_wait_ld();
        const int n = n0 + c;
        if (!row_ok || n >= pr.N) continue;
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        const long long off = row_off + (long long)(n / pr.cols_per_group) * pr.s_group_col +
                              (n % pr.cols_per_group);
        if (n + 32 <= pr.N && (n % pr.cols_per_group) + 32 <= pr.cols_per_group) {
          uint4* dst = reinterpret_cast<uint4*>(out + off);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        } else {
          for (int j = 0; j < 32 && n + j < pr.N; ++j) {
            const int nn = n + j;
            const long long o = row_off + (long long)(nn / pr.cols_per_group) * pr.s_group_col +
                                (nn % pr.cols_per_group);
            const uint32_t word = pk[j >> 1];
            const uint16_t bits = (j & 1) ? (uint16_t)(word >> 16) : (uint16_t)(word & 0xFFFF);
            out[o] = __ushort_as_bfloat16(bits);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  // Every lane of a warp meets here before the CTA-wide barrier: a barrier
  // counts whole warps, so a warp must not reach it split across branches.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int BN>
mha_status launch(GemmTcParams& P, cudaStream_t s) {
  using C = Cfg<BN>;
  int total = 0;
  P.tile_start[0] = 0;
  for (int i = 0; i < P.nprob; ++i) {
    P.tiles_n[i] = (P.prob[i].N + BN - 1) / BN;
    total += ((P.prob[i].M + BM - 1) / BM) * P.tiles_n[i];
    P.tile_start[i + 1] = total;
  }
  for (int i = P.nprob; i < MAXP; ++i) P.tile_start[i + 1] = total;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM) != cudaSuccess)
      return MHA_ERR_CUDA;
    attr_set = true;
  }
  const int grid = total < num_sms() ? total : num_sms();
  const cudaError_t e = launch_dependent(gemm_tc_kernel<BN>, dim3(grid), dim3(192), C::SMEM, s, P);
  count_launch();
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace

mha_status gemm_tc(const GemmProblem* probs, int nprob, int32_t* err, cudaStream_t s) {
  if (nprob < 1 || nprob > MAXP) return MHA_ERR_INVALID_ARG;
  GemmTcParams P;
  memset(&P, 0, sizeof(P));
  P.nprob = nprob;
  P.err = err;
  P.limit_ns = wait_limit_ns();
  bool all256 = true;
  for (int i = 0; i < nprob; ++i) {
    const GemmProblem& pr = probs[i];
    P.prob[i] = pr;
    if (pr.N % 256) all256 = false;
    // A: row-major M x K (K contiguous).
    const uint64_t adims[2] = {(uint64_t)pr.K, (uint64_t)pr.M};
    const uint64_t astr[1] = {(uint64_t)pr.K * 2};
    const uint32_t abox[2] = {64, BM};
    // W: row-major K x N (N contiguous), loaded as 64-column panels.
    const uint64_t bdims[2] = {(uint64_t)pr.N, (uint64_t)pr.K};
    const uint64_t bstr[1] = {(uint64_t)pr.N * 2};
    const uint32_t bbox[2] = {64, BK};
    if (!make_tmap_bf16(&P.amap[i], pr.A, 2, adims, astr, abox, true) ||
        !make_tmap_bf16(&P.bmap[i], pr.W, 2, bdims, bstr, bbox, true))
      return MHA_ERR_CUDA;
    // 16-byte vector stores in the epilogue: every row pitch, group stride and
    // 32-column chunk offset is a multiple of 8 elements
    if (pr.cols_per_group % 8 || pr.N % 8 || pr.s_row % 8 || pr.s_group_col % 8 ||
        pr.s_group_row % 8)
      return MHA_ERR_UNSUPPORTED;
  }
  return all256 ? launch<256>(P, s) : launch<128>(P, s);
}

}  // namespace mha
