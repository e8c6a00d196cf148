// attn_tc.cu - fused masked attention on tcgen05 tensor cores (bf16).
//
// For one (batch item b, head i, 128-row query tile) a CTA folds the allowed
// keys block by block into the stable summary of every query row ("Stable
// summary of an attention key block", Definition, alphabetamath.cc):
//   m = max_j s_ij,  l = sum_j e^{s_ij - m},  z = sum_j e^{s_ij - m} v_j
// merging each 128-key block's summary into the running one with
//   m' = max(m, m_blk),  l' = e^{m - m'} l + e^{m_blk - m'} l_blk,  z' likewise,
// and writes z / l once per row. The n_q x n_k score matrix only ever exists
// one 128 x 128 block at a time, in tensor memory.
//
// Roles (192 threads):
//   warp 0      TMA producer: Q once, then K and V blocks into a STAGES ring
//   warp 1      MMA issuer: S_j = Q K_j^T (SMEM x SMEM -> TMEM), then
//               z += P_j V_j (P from TMEM, V from SMEM -> TMEM accumulator O)
//   warps 2..5  softmax: thread = query row = TMEM lane. Loads its row of S_j,
//               takes the row max in-thread (no shuffles: a TMEM lane holds a
//               whole row), computes p = 2^{c log2(e) s - m}, its sum, writes p
//               as bf16 into the columns of S_j (P aliases S), and rescales its
//               row of O by e^{m - m'} only when its max grew. At the end:
//               O / l -> bf16 -> Z in the concatenated (B, n_q, h*d_vh) layout.
// S is double-buffered in TMEM so S_{j+1} = Q K_{j+1}^T runs while the
// softmax works on S_j. Fully masked key blocks (past the diagonal, past the
// valid length) are never loaded: they are the empty summary.
#include <cuda_bf16.h>
#include <math.h>

#include "device_common.cuh"
#include "internal.h"

namespace mha {
namespace {

constexpr int BLK_M = 128;  // query rows per CTA
constexpr int BLK_N = 128;  // keys per block
constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL = 256, TMEM_COLS = 512;

struct AttnTcParams {
  CUtensorMap qmap;  // Q: dims {d_h, n_q, B*h}, box {64, 128, 1}
  CUtensorMap kmap;  // K: dims {d_h, n_k, B*h}, box {64, 128, 1}
  CUtensorMap vmap;  // V: dims {d_vh, n_k, B*h}, box {64, 128, 1}
  void* Z;
  int n_q, n_k, h;
  float cl2;         // |c| * log2(e)
  int negate;        // c < 0: S is computed as -Q K^T (MMA negate-A bit)
  int causal, padding, pad_queries;
  int32_t* err;
  uint64_t limit_ns;
  int valid_len[MHA_MAX_PADDED_BATCH];
};

template <int DQK, int DV>
struct ACfg {
  static constexpr int Q_BYTES = BLK_M * DQK * 2;
  static constexpr int K_BYTES = BLK_N * DQK * 2;
  static constexpr int V_BYTES = BLK_N * DV * 2;
  static constexpr int STAGES = (DQK + DV) <= 192 ? 3 : 2;
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
  static constexpr int SMEM = Q_BYTES + STAGES * STAGE_BYTES + 1024 + 256;
};

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if (globaltimer_ns() - t0 > 100000000ull) return;
  }
}

template <int DQK, int DV>
__global__ void __launch_bounds__(192, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams P) {
  using C = ACfg<DQK, DV>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_qt = gridDim.x;
  // causal: heavy tiles (large q0) first, so the light ones fill the tail
  const int qt = P.causal ? (n_qt - 1 - (int)blockIdx.x) : (int)blockIdx.x;
  const int q0 = qt * BLK_M;
  const int head = blockIdx.y, b = blockIdx.z;
  const int L = P.padding ? P.valid_len[b] : P.n_k;
  const int q_end = P.pad_queries ? min(L, P.n_q) : P.n_q;
  int k_end = L;
  if (P.causal) k_end = min(k_end, q0 + BLK_M);
  const int nblk = (q0 < q_end) ? (k_end + BLK_N - 1) / BLK_N : 0;
  __nv_bfloat16* Zg = static_cast<__nv_bfloat16*>(P.Z);
  const long long zrow_stride = (long long)P.h * DV;
  const long long zbase = (long long)b * P.n_q * zrow_stride + (long long)head * DV;

  if (nblk == 0) {
    // every row of this tile is padding: Z rows are exact zeros
    const int rows = min(BLK_M, P.n_q - q0);
    for (int e = threadIdx.x; e < rows * (DV / 8); e += blockDim.x) {
      const int r = e / (DV / 8), c8 = e % (DV / 8);
      *reinterpret_cast<uint4*>(Zg + zbase + (long long)(q0 + r) * zrow_stride + c8 * 8) =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + C::Q_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(kv_s + C::STAGES * C::STAGE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;            // [STAGES]
  uint64_t* v_full = k_full + C::STAGES;    // [STAGES]
  uint64_t* k_empty = v_full + C::STAGES;   // [STAGES] freed by S = Q K^T
  uint64_t* v_empty = k_empty + C::STAGES;  // [STAGES] freed by z += P V
  uint64_t* s_full = v_empty + C::STAGES;   // [2]
  uint64_t* p_full = s_full + 2;            // [2]
  uint64_t* o_full = p_full + 2;            // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_full + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);  // one arrival per softmax warp
    }
    mbar_init(o_full, 1);
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
  const WaitCtl w{P.err, abort_flag, P.limit_ns};
  const int bh = b * P.h + head;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&P.qmap);
      tma_prefetch_desc(&P.kmap);
      tma_prefetch_desc(&P.vmap);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int p = 0; p < DQK / 64; ++p) tma_load_3d(q_s + p * 16384, &P.qmap, q_full, 64 * p, q0, bh);
      int kb = 0;
      bool gave_up = false;
      for (; kb < nblk; ++kb) {
        const int s = kb % C::STAGES;
        uint8_t* k_s = kv_s + s * C::STAGE_BYTES;
        uint8_t* v_s = k_s + C::K_BYTES;
        const int k0 = kb * BLK_N;
        const uint32_t reuse = ((kb / C::STAGES) - 1) & 1;
        if (kb >= C::STAGES && !mbar_wait(&k_empty[s], reuse, w)) {
          gave_up = true;
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], C::K_BYTES);
#pragma unroll
        for (int p = 0; p < DQK / 64; ++p)
          tma_load_3d(k_s + p * 16384, &P.kmap, &k_full[s], 64 * p, k0, bh);
        if (kb >= C::STAGES && !mbar_wait(&v_empty[s], reuse, w)) {
          ++kb;  // K of this block is in flight: drain it too
          gave_up = true;
          break;
        }
        mbar_arrive_expect_tx(&v_full[s], C::V_BYTES);
#pragma unroll
        for (int p = 0; p < DV / 64; ++p)
          tma_load_3d(v_s + p * 16384, &P.vmap, &v_full[s], 64 * p, k0, bh);
      }
      if (gave_up) {  // let this CTA's loads land before it exits
        drain(q_full, 0);
        for (int k = (kb > C::STAGES ? kb - C::STAGES : 0); k < kb; ++k) {
          drain(&k_full[k % C::STAGES], (k / C::STAGES) & 1);
          drain(&v_full[k % C::STAGES], (k / C::STAGES) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(BLK_M, BLK_N, 0, 0) | (P.negate ? (1u << 13) : 0u);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BLK_M, DV, 0, 1);
      const uint32_t q_addr = smem_u32(q_s);
      bool ok = mbar_wait(q_full, 0, w);
      auto issue_s = [&](int kb) -> bool {
        const int s = kb % C::STAGES;
        if (!mbar_wait(&k_full[s], (kb / C::STAGES) & 1, w)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(kv_s + s * C::STAGE_BYTES);
        const uint32_t d = tmem + ((kb & 1) ? S_COL1 : S_COL0);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
          umma_ss(d, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                  idesc_qk, kk > 0);
        }
        umma_commit(&k_empty[s]);  // this K stage can be refilled once S_kb is done
        umma_commit(&s_full[kb & 1]);
        return true;
      };
      auto issue_pv = [&](int kb) -> bool {
        const int s = kb % C::STAGES;
        if (!mbar_wait(&p_full[kb & 1], (kb >> 1) & 1, w)) return false;
        if (!mbar_wait(&v_full[s], (kb / C::STAGES) & 1, w)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(kv_s + s * C::STAGE_BYTES + C::K_BYTES);
        const uint32_t p_tmem = tmem + ((kb & 1) ? S_COL1 : S_COL0);
#pragma unroll
        for (int kk = 0; kk < BLK_N / 16; ++kk) {
          // V is MN-major: 16 key rows of 128 B; 64-column panels 16 KB apart.
          umma_ts(tmem + O_COL, p_tmem + kk * 8, sdesc_sw128(v_addr + kk * 2048, 16384, 1024),
                  idesc_pv, (kb > 0 || kk > 0));
        }
        umma_commit(&v_empty[s]);
        umma_commit(o_full);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int kb = 0; kb < nblk && ok; ++kb) {
        if (kb + 1 < nblk) ok = issue_s(kb + 1);
        if (ok) ok = issue_pv(kb);
      }
      if (!ok) {  // gave up: wait for this thread's MMAs before TMEM is released
        umma_commit(&s_full[0]);
        drain(&s_full[0], 0);
        drain(&s_full[0], 1);
      }
    }
  } else {
    // Softmax warps: warp w owns TMEM lanes (query rows) 32*(w%4) .. +31.
    const int g = warp & 3;
    const int r = 32 * g + lane;
    const int q = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(32 * g) << 16;
    const float cl2 = P.cl2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int kb = 0; kb < nblk; ++kb) {
      if (!mbar_wait(&s_full[kb & 1], (kb >> 1) & 1, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_off + ((kb & 1) ? S_COL1 : S_COL0);
      uint32_t sr[BLK_N];
#pragma unroll
      for (int c = 0; c < BLK_N / 32; ++c)
        tmem_ld32(s_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tmem_wait_ld();
      const int k0 = kb * BLK_N;
      const bool masked = (k0 + BLK_N > L) || (P.causal && k0 + BLK_N - 1 > q0);
      // allowed keys of this row in this block: k0 + c < lim
      const int lim = masked ? (P.causal ? min(L, q + 1) : L) - k0 : BLK_N;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BLK_N; ++c)
        mx = fmaxf(mx, (!masked || c < lim) ? __uint_as_float(sr[c]) : -INFINITY);
      const float m_blk = (mx == -INFINITY) ? -INFINITY : mx * cl2;
      const float m_new = fmaxf(m_run, m_blk);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - m_use);  // e^{m - m'}; 0 when m = -inf
      float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
      uint32_t pk[BLK_N / 2];
#pragma unroll
      for (int c = 0; c < BLK_N; c += 4) {
        float p0 = ex2_approx(fmaf(__uint_as_float(sr[c + 0]), cl2, -m_use));
        float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), cl2, -m_use));
        float p2 = ex2_approx(fmaf(__uint_as_float(sr[c + 2]), cl2, -m_use));
        float p3 = ex2_approx(fmaf(__uint_as_float(sr[c + 3]), cl2, -m_use));
        if (masked) {  // forbidden keys get weight exactly 0
          p0 = (c + 0 < lim) ? p0 : 0.f;
          p1 = (c + 1 < lim) ? p1 : 0.f;
          p2 = (c + 2 < lim) ? p2 : 0.f;
          p3 = (c + 3 < lim) ? p3 : 0.f;
        }
        sum0 += p0;
        sum1 += p1;
        sum2 += p2;
        sum3 += p3;
        pk[c / 2] = pack_bf16x2(p0, p1);
        pk[c / 2 + 1] = pack_bf16x2(p2, p3);
      }
      l_run = l_run * alpha + ((sum0 + sum1) + (sum2 + sum3));
      // P_j overwrites the first BLK_N/2 columns of S_j (two bf16 per column)
      tmem_st32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      // merge into the running summary: rescale this row of O by e^{m - m'}
      // when its max grew (O must hold every earlier block first)
      const bool grow = kb > 0 && m_new > m_run;
      if (__any_sync(0xffffffffu, grow)) {
        if (!mbar_wait(o_full, (kb - 1) & 1, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t o_addr = tmem + lane_off + O_COL;
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st32(o_addr + 32 * c, o);
        }
      }
      m_run = m_new;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[kb & 1]);
    }
    if (ok && mbar_wait(o_full, (nblk - 1) & 1, w)) {
      tc_fence_after();
      const bool computed = q < q_end;
      const float inv = computed ? 1.f / l_run : 0.f;
      const uint32_t o_addr = tmem + lane_off + O_COL;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(o_addr + 32 * c, o);
        tmem_wait_ld();
        if (q < P.n_q) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = computed ? pack_bf16x2(__uint_as_float(o[2 * j]) * inv,
                                           __uint_as_float(o[2 * j + 1]) * inv)
                             : 0u;
          uint4* dst = reinterpret_cast<uint4*>(Zg + zbase + (long long)q * zrow_stride + 32 * c);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int DQK, int DV>
mha_status launch(const AttnTcParams& P, int B, int h, int n_q, cudaStream_t s) {
  using C = ACfg<DQK, DV>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_tc_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM) != cudaSuccess)
      return MHA_ERR_CUDA;
    attr = true;
  }
  const dim3 grid((n_q + BLK_M - 1) / BLK_M, h, B);
  attn_tc_kernel<DQK, DV><<<grid, 192, C::SMEM, s>>>(P);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace

mha_status attention_tc(const AttnArgs& a, cudaStream_t s) {
  if (a.h > 65535 || a.B > 65535) return MHA_ERR_UNSUPPORTED;
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
  P.n_q = a.n_q;
  P.n_k = a.n_k;
  P.h = a.h;
  P.cl2 = fabsf(a.c) * 1.4426950408889634f;
  P.negate = a.c < 0.f;
  P.causal = a.causal;
  P.padding = a.padding;
  P.pad_queries = a.pad_queries;
  P.err = a.err;
  P.limit_ns = wait_limit_ns();
  for (int b = 0; b < MHA_MAX_PADDED_BATCH; ++b)
    P.valid_len[b] = (a.padding && b < a.B) ? a.valid_len_host[b] : a.n_k;
  if (a.d_h == 64 && a.d_vh == 64) return launch<64, 64>(P, a.B, a.h, a.n_q, s);
  if (a.d_h == 128 && a.d_vh == 128) return launch<128, 128>(P, a.B, a.h, a.n_q, s);
  if (a.d_h == 64 && a.d_vh == 128) return launch<64, 128>(P, a.B, a.h, a.n_q, s);
  if (a.d_h == 128 && a.d_vh == 64) return launch<128, 64>(P, a.B, a.h, a.n_q, s);
  return MHA_ERR_UNSUPPORTED;
}

}  // namespace mha
