// decode.cu - attention of a few query rows over a long key/value cache,
// split over the keys and merged with the summary merge.
//
// "Stable summary of an attention key block" (alphabetamath.cc, Definition):
// the summary (m, l, z) of a key set, and the merge of the summaries of two
// disjoint sets, m' = max(m_S, m_T), l' = e^{m_S - m'} l_S + e^{m_T - m'} l_T,
// z' likewise; z / l of the merged summary is the attention output over the
// union. Here the keys of one (batch item, head) are cut into chunks of
// DEC_CHUNK keys and each warp of a chunk's CTA folds a share of them, 32 at a
// time, into its own summary (pass 1); pass 2 merges every partial summary of
// a query row and writes z / l. Summaries are kept in base 2: scores are
// pre-multiplied by c log2(e), which leaves z / l unchanged.
//
// The work is bound by reading K and V once (a handful of query rows), so it
// runs on CUDA cores: lane j of a warp scores key j of a 32-key group against
// every query row, the group's weights are shuffled across the lanes, and
// each lane accumulates its own columns of z.
#include <cuda_bf16.h>
#include <math.h>

#include "device_common.cuh"
#include "internal.h"

namespace mha {
namespace {

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
#ifndef MHA_DECODE_CHUNK
#define MHA_DECODE_CHUNK 1024
#endif
constexpr int DEC_CHUNK = MHA_DECODE_CHUNK;  // keys per CTA
constexpr int DEC_NQ = 8;       // query rows per pass over the chunk
#ifndef MHA_DECODE_VUNROLL
#define MHA_DECODE_VUNROLL 4
#endif
constexpr int DEC_VUNROLL = MHA_DECODE_VUNROLL;  // value rows in flight per lane

struct DecodeParams {
  const void* Q;   // (B, h, n_q, d_h)
  const void* K;   // (B, h, n_k, d_h)
  const void* V;   // (B, h, n_k, d_vh)
  void* Z;         // (B, n_q, h * d_vh)
  float* part;     // [B][h][n_q][nsplit][2 + d_vh]: m, l, z of each warp's keys
  int B, n_q, n_k, h, d_h, d_vh, nsplit;
  float cl2;       // c * log2(e)
  int causal_tail; // row i sees keys j <= L - n_q + i
  int valid_len[MHA_MAX_PADDED_BATCH];
  // the streaming kernel's work: the 32-key groups of every (batch item,
  // head) key sequence, numbered batch item by batch item, head by head;
  // item_start[b] = first group of batch item b, nitems = all groups. CTA c
  // of G takes groups [c nitems / G, (c + 1) nitems / G).
  int nitems;
  int item_start[MHA_MAX_PADDED_BATCH + 1];
  // summaries per DEC_CHUNK keys: DEC_WARPS (one per warp of pass 1), or 1
  // (the streaming kernel combines its warps' summaries of a chunk first)
  int per_chunk;
  uint64_t limit_ns;  // bounded waits give up after this long
};

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// Eight consecutive elements starting at a 16-byte aligned address.
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ float dwarp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float dwarp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Pass 1. grid (chunks, h, B). Warp w of chunk ch folds the keys
// k0 + 32 (w + DEC_WARPS it) + lane, it = 0, 1, ... (below the chunk end and
// the valid length) into one summary per query row, and writes it as split
// ch * DEC_WARPS + w. VW: z columns per lane (d_vh <= 32 VW). VEC: d_h is a
// multiple of 8 and K rows are 16-byte aligned (vector loads).
template <typename T, int VW, bool VEC>
__global__ void __launch_bounds__(DEC_THREADS) decode_partial_kernel(
    const __grid_constant__ DecodeParams P) {
  __shared__ __align__(16) float qs[DEC_NQ][256];
  const int chunk = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int L = P.valid_len[b];
  const int k0 = chunk * DEC_CHUNK;
  if (k0 >= L) return;  // the merge reads only the splits below L
  const int k1 = min(L, k0 + DEC_CHUNK);
  const int dq = P.d_h, dv = P.d_vh;
  const long long bh = (long long)b * P.h + head;
  const T* Qg = static_cast<const T*>(P.Q) + bh * P.n_q * dq;
  const T* Kg = static_cast<const T*>(P.K) + bh * P.n_k * dq;
  const T* Vg = static_cast<const T*>(P.V) + bh * P.n_k * dv;
  const int split = chunk * DEC_WARPS + warp;

  for (int r0 = 0; r0 < P.n_q; r0 += DEC_NQ) {
    const int nr = min(DEC_NQ, P.n_q - r0);
    __syncthreads();
    for (int e = threadIdx.x; e < nr * dq; e += DEC_THREADS) {
      const int r = e / dq, k = e % dq;
      qs[r][k] = ldf(Qg + (long long)(r0 + r) * dq + k) * P.cl2;
    }
    __syncthreads();
    float m_run[DEC_NQ], l_run[DEC_NQ], z_run[DEC_NQ][VW];
#pragma unroll
    for (int r = 0; r < DEC_NQ; ++r) {
      m_run[r] = -INFINITY;
      l_run[r] = 0.f;
#pragma unroll
      for (int t = 0; t < VW; ++t) z_run[r][t] = 0.f;
    }
    for (int g0 = k0 + 32 * warp; g0 < k1; g0 += 32 * DEC_WARPS) {
      const int key = g0 + lane;
      const bool in = key < k1;
      // scores of this lane's key against every query row (already in log2 units)
      float s[DEC_NQ];
#pragma unroll
      for (int r = 0; r < DEC_NQ; ++r) s[r] = 0.f;
      if (in) {
        const T* krow = Kg + (long long)key * dq;
        if (VEC) {
          // 8 elements per 16-byte load (two for fp32); rows are 16-byte aligned
          for (int k = 0; k < dq; k += 8) {
            float kv[8];
            load8(krow + k, kv);
#pragma unroll
            for (int r = 0; r < DEC_NQ; ++r) {
              const float4 q0 = *reinterpret_cast<const float4*>(&qs[r][k]);
              const float4 q1 = *reinterpret_cast<const float4*>(&qs[r][k + 4]);
              float acc = s[r];
              acc = fmaf(q0.x, kv[0], acc);
              acc = fmaf(q0.y, kv[1], acc);
              acc = fmaf(q0.z, kv[2], acc);
              acc = fmaf(q0.w, kv[3], acc);
              acc = fmaf(q1.x, kv[4], acc);
              acc = fmaf(q1.y, kv[5], acc);
              acc = fmaf(q1.z, kv[6], acc);
              acc = fmaf(q1.w, kv[7], acc);
              s[r] = acc;
            }
          }
        } else {
          for (int k = 0; k < dq; ++k) {
            const float kv = ldf(krow + k);
#pragma unroll
            for (int r = 0; r < DEC_NQ; ++r) s[r] = fmaf(qs[r][k], kv, s[r]);
          }
        }
      }
      float p[DEC_NQ];
#pragma unroll
      for (int r = 0; r < DEC_NQ; ++r) {
        p[r] = 0.f;
        if (r >= nr) continue;  // uniform
        bool allowed = in;
        if (P.causal_tail) allowed = allowed && key <= L - P.n_q + r0 + r;
        const float sv = allowed ? s[r] : -INFINITY;
        const float m_blk = dwarp_max(sv);
        if (m_blk == -INFINITY) continue;  // no allowed key in this group: the empty summary
        // merge the group's summary into the running one (base 2)
        const float m_new = fmaxf(m_run[r], m_blk);
        const float a = exp2f(m_run[r] - m_new);
        p[r] = allowed ? exp2f(sv - m_new) : 0.f;
        l_run[r] = l_run[r] * a + dwarp_sum(p[r]);
#pragma unroll
        for (int t = 0; t < VW; ++t) z_run[r][t] *= a;
        m_run[r] = m_new;
      }
      // z += sum over the group's keys of p_j v_j; lane owns columns lane + 32 t
      const int ng = min(32, k1 - g0);
      for (int j = 0; j < ng; ++j) {
        const T* vrow = Vg + (long long)(g0 + j) * dv;
        float vv[VW];
#pragma unroll
        for (int t = 0; t < VW; ++t) {
          const int col = lane + 32 * t;
          vv[t] = col < dv ? ldf(vrow + col) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < DEC_NQ; ++r) {
          const float pj = __shfl_sync(0xffffffffu, p[r], j);
#pragma unroll
          for (int t = 0; t < VW; ++t) z_run[r][t] = fmaf(pj, vv[t], z_run[r][t]);
        }
      }
    }
    // this warp's summaries of the group of rows
#pragma unroll
    for (int r = 0; r < DEC_NQ; ++r) {
      if (r >= nr) continue;
      float* dst = P.part + ((bh * P.n_q + r0 + r) * P.nsplit + split) * (long long)(2 + dv);
      if (lane == 0) {
        dst[0] = m_run[r];
        dst[1] = l_run[r];
      }
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        const int col = lane + 32 * t;
        if (col < dv) dst[2 + col] = z_run[r][t];
      }
    }
  }
}

// Raw words of a 16-byte chunk and their values: 8 bf16 or 4 fp32.
template <typename T>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& u, float* v) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& u, float* v) {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
  }
};

// DV / 32 consecutive values of a row, as a lane's share of a warp-wide load.
template <typename T, int CPL>
__device__ __forceinline__ void load_cols(const T* p, float (&v)[CPL]) {
  if constexpr (sizeof(T) == 2) {
    static_assert(CPL == 2 || CPL == 4 || CPL == 8, "columns per lane");
    if constexpr (CPL == 2) {
      const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
      v[0] = __uint_as_float(u << 16);
      v[1] = __uint_as_float(u & 0xffff0000u);
    } else if constexpr (CPL == 4) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
      v[0] = __uint_as_float(u.x << 16);
      v[1] = __uint_as_float(u.x & 0xffff0000u);
      v[2] = __uint_as_float(u.y << 16);
      v[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
      Vec16<__nv_bfloat16>::unpack(u, v);
    }
  } else {
    static_assert(CPL == 2 || CPL == 4, "columns per lane");
    if constexpr (CPL == 2) {
      const float2 u = __ldg(reinterpret_cast<const float2*>(p));
      v[0] = u.x;
      v[1] = u.y;
    } else {
      const float4 u = __ldg(reinterpret_cast<const float4*>(p));
      v[0] = u.x;
      v[1] = u.y;
      v[2] = u.z;
      v[3] = u.w;
    }
  }
}

// W consecutive 32-bit words at a 4 W-byte aligned address, in one load.
template <int W>
__device__ __forceinline__ void load_words(const void* p, uint32_t (&w)[W]) {
  static_assert(W == 1 || W == 2 || W == 4, "words per load");
  if constexpr (W == 1) {
    w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
  } else if constexpr (W == 2) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = u.x;
    w[1] = u.y;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = u.x;
    w[1] = u.y;
    w[2] = u.z;
    w[3] = u.w;
  }
}

// The CPL values held in the raw words of one load_words.
template <typename T, int CPL, int W>
__device__ __forceinline__ void unpack_words(const uint32_t (&w)[W], float (&v)[CPL]) {
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int i = 0; i < W; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = __uint_as_float(w[i]);
  }
}

// Pass 1 for head sizes known at compile time (d_h = DQK, d_vh = DV, both
// multiples of 32 and of 8 elements per 16 bytes), NQ query rows per pass.
// A lane issues every load of its key row before using any of them, and the
// value rows are read as warp-wide vectors (lane owns columns
// [lane*DV/32, (lane+1)*DV/32)); for a full group of 32 keys the value rows
// are requested together with the key rows, before any arithmetic, so the
// whole group (32 K rows and 32 V rows) is in flight per warp at once.
template <typename T, int NQ, int DQK, int DV>
__global__ void __launch_bounds__(DEC_THREADS) decode_partial_fast_kernel(
    const __grid_constant__ DecodeParams P) {
  constexpr int CPL = DV / 32;           // z columns per lane
  constexpr int KV16 = DQK / Vec16<T>::N; // 16-byte chunks per key row
  constexpr int VW = CPL * (int)sizeof(T) / 4;  // 32-bit words of a lane's share of a V row
  // value rows requested with the key rows when both fit in registers
  constexpr bool V_AHEAD = 32 * VW + 4 * KV16 <= 128;
  __shared__ __align__(16) float qs[NQ][DQK];
  const int chunk = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int L = P.valid_len[b];
  const int k0 = chunk * DEC_CHUNK;
  if (k0 >= L) return;
  const int k1 = min(L, k0 + DEC_CHUNK);
  const long long bh = (long long)b * P.h + head;
  const T* Qg = static_cast<const T*>(P.Q) + bh * P.n_q * DQK;
  const T* Kg = static_cast<const T*>(P.K) + bh * P.n_k * DQK;
  const T* Vg = static_cast<const T*>(P.V) + bh * P.n_k * DV;
  const int split = chunk * DEC_WARPS + warp;

  for (int r0 = 0; r0 < P.n_q; r0 += NQ) {
    const int nr = min(NQ, P.n_q - r0);
    __syncthreads();
    for (int e = threadIdx.x; e < NQ * DQK; e += DEC_THREADS) {
      const int r = e / DQK, k = e % DQK;
      qs[r][k] = r < nr ? ldf(Qg + (long long)(r0 + r) * DQK + k) * P.cl2 : 0.f;
    }
    __syncthreads();
    float m_run[NQ], l_run[NQ], z_run[NQ][CPL];
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      m_run[r] = -INFINITY;
      l_run[r] = 0.f;
#pragma unroll
      for (int t = 0; t < CPL; ++t) z_run[r][t] = 0.f;
    }
    for (int g0 = k0 + 32 * warp; g0 < k1; g0 += 32 * DEC_WARPS) {
      const int key = g0 + lane;
      const bool in = key < k1;
      const bool full = V_AHEAD && g0 + 32 <= k1;  // uniform across the warp
      const T* vbase = Vg + (long long)g0 * DV + lane * CPL;
      float s[NQ];
#pragma unroll
      for (int r = 0; r < NQ; ++r) s[r] = 0.f;
      uint32_t vraw[V_AHEAD ? 32 : 1][VW];
      if (in) {
        const uint4* krow = reinterpret_cast<const uint4*>(Kg + (long long)key * DQK);
        uint4 raw[KV16];
#pragma unroll
        for (int i = 0; i < KV16; ++i) raw[i] = __ldg(krow + i);
        if constexpr (V_AHEAD) {
          if (full) {
#pragma unroll
            for (int j = 0; j < 32; ++j) load_words<VW>(vbase + (long long)j * DV, vraw[j]);
          }
        }
#pragma unroll
        for (int i = 0; i < KV16; ++i) {
          float kv[Vec16<T>::N];
          Vec16<T>::unpack(raw[i], kv);
#pragma unroll
          for (int r = 0; r < NQ; ++r) {
#pragma unroll
            for (int e = 0; e < Vec16<T>::N; ++e)
              s[r] = fmaf(qs[r][i * Vec16<T>::N + e], kv[e], s[r]);
          }
        }
      }
      float p[NQ];
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        p[r] = 0.f;
        if (r >= nr) continue;  // uniform
        bool allowed = in;
        if (P.causal_tail) allowed = allowed && key <= L - P.n_q + r0 + r;
        const float sv = allowed ? s[r] : -INFINITY;
        const float m_blk = dwarp_max(sv);
        if (m_blk == -INFINITY) continue;  // the empty summary
        const float m_new = fmaxf(m_run[r], m_blk);
        const float a = exp2f(m_run[r] - m_new);
        p[r] = allowed ? exp2f(sv - m_new) : 0.f;
        l_run[r] = l_run[r] * a + dwarp_sum(p[r]);
#pragma unroll
        for (int t = 0; t < CPL; ++t) z_run[r][t] *= a;
        m_run[r] = m_new;
      }
      if (full) {
#pragma unroll
        for (int j = 0; j < (V_AHEAD ? 32 : 0); ++j) {
          float vv[CPL];
          unpack_words<T, CPL, VW>(vraw[j], vv);
#pragma unroll
          for (int r = 0; r < NQ; ++r) {
            const float pj = __shfl_sync(0xffffffffu, p[r], j);
#pragma unroll
            for (int t = 0; t < CPL; ++t) z_run[r][t] = fmaf(pj, vv[t], z_run[r][t]);
          }
        }
      } else {
        const int ng = k1 - g0;
#pragma unroll DEC_VUNROLL
        for (int j = 0; j < ng; ++j) {
          float vv[CPL];
          load_cols<T, CPL>(vbase + (long long)j * DV, vv);
#pragma unroll
          for (int r = 0; r < NQ; ++r) {
            const float pj = __shfl_sync(0xffffffffu, p[r], j);
#pragma unroll
            for (int t = 0; t < CPL; ++t) z_run[r][t] = fmaf(pj, vv[t], z_run[r][t]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      if (r >= nr) continue;
      float* dst = P.part + ((bh * P.n_q + r0 + r) * P.nsplit + split) * (long long)(2 + DV);
      if (lane == 0) {
        dst[0] = m_run[r];
        dst[1] = l_run[r];
      }
#pragma unroll
      for (int t = 0; t < CPL; ++t) dst[2 + lane * CPL + t] = z_run[r][t];
    }
  }
}

// ---------------------------------------------------------------------------
// Streaming pass 1 (bf16, d_h = d_vh = D in {64, 128}, up to 8 query rows).
//
// One CTA per SM takes an equal contiguous range of the 32-key groups of all
// (batch item, head) sequences and walks it piece by piece (a piece: its
// groups of one DEC_CHUNK-key chunk of one sequence). One producer thread
// copies each group of the cache, its K rows and its V rows (contiguous in the
// head-split layout), into a DS_STAGES-deep shared-memory ring with bulk
// asynchronous copies, as far ahead as the ring allows and independently of
// the arithmetic, so that many groups' bytes are in flight per SM. Consumer
// warp w takes groups n = w, w + DS_WARPS, ... of the CTA's sequence and folds
// each into its own summary of the piece's rows; at the end of a piece the
// warps' summaries are merged through shared memory and written once, into
// the chunk's first or second slot (see DsPiece).
// ---------------------------------------------------------------------------

constexpr int DS_WARPS = DEC_WARPS;  // consumer warps: same split count as pass 1
constexpr int DS_THREADS = 32 * (DS_WARPS + 1);
constexpr int DS_STAGES = 12;

template <int NQ, int D>
struct DsCfg {
  static constexpr int ROW = D * 2;               // bytes of one K or V row
  static constexpr int STAGE = 2 * 32 * ROW;      // K rows then V rows of a group
  static constexpr int Q_FLOATS = NQ * D;         // one item's rows, fp32, pre-scaled
  // the combine of the warps' summaries of a chunk: m and l of each warp,
  // then each warp's weighted z
  static constexpr int COMBINE_FLOATS = 2 * DS_WARPS + DS_WARPS * D;
  static constexpr int SMEM =
      DS_STAGES * STAGE + 2 * Q_FLOATS * 4 + 2 * DS_STAGES * 8 + 16 + COMBINE_FLOATS * 4;
};

constexpr int DS_GROUP = 32;                       // keys per group (one per lane)
constexpr int DS_CHUNK_GROUPS = DEC_CHUNK / DS_GROUP;  // groups per summary chunk
static_assert(DEC_CHUNK % DS_GROUP == 0, "chunk of whole groups");

// A piece of a CTA's group range: keys [k0, k1) of the (b, head) sequence,
// inside one chunk. Its summary goes to slot 2 chunk (the piece that starts
// the chunk) or 2 chunk + 1 (the rest of a chunk that a range boundary cut);
// a piece that is its whole chunk also marks slot 2 chunk + 1 empty. Every
// range holds at least a chunk's worth of groups, so no chunk has more than
// two pieces.
struct DsPiece {
  int b, head, chunk, k0, k1, slot;
  bool clear_rest;
};

// The next piece from group g (advanced past it) of a range ending at g_end.
__device__ __forceinline__ bool ds_next_piece(const DecodeParams& P, int& g, int g_end,
                                              DsPiece& pc) {
  if (g >= g_end) return false;
  int lo = 0, hi = P.B - 1;
  while (lo < hi) {  // last b with item_start[b] <= g
    const int mid = (lo + hi + 1) >> 1;
    if (P.item_start[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  const int L = P.valid_len[lo];
  const int ng = (L + DS_GROUP - 1) / DS_GROUP;  // groups of one head's sequence
  const int local = g - P.item_start[lo];
  const int gi = local % ng;
  pc.b = lo;
  pc.head = local / ng;
  pc.chunk = gi / DS_CHUNK_GROUPS;
  const int cstart = pc.chunk * DS_CHUNK_GROUPS;
  const int cend = min(ng, cstart + DS_CHUNK_GROUPS);
  const int len = min(cend - gi, g_end - g);
  pc.k0 = gi * DS_GROUP;
  pc.k1 = min(L, (gi + len) * DS_GROUP);
  pc.slot = 2 * pc.chunk + (gi == cstart ? 0 : 1);
  pc.clear_rest = gi == cstart && gi + len == cend;
  g += len;
  return true;
}

// A bounded wait that ignores the abort flag: used only while draining copies
// this CTA itself started, before it exits.
__device__ __forceinline__ void ds_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if (globaltimer_ns() - t0 > 100000000ull) return;  // 100 ms
  }
}

template <int NQ, int D>
__global__ void __launch_bounds__(DS_THREADS, 1) decode_stream_kernel(
    const __grid_constant__ DecodeParams P) {
  using C = DsCfg<NQ, D>;
  constexpr int CPL = D / 32;  // z columns per lane
  constexpr int NCH = D / 8;   // 16-byte chunks of a row
  extern __shared__ __align__(1024) uint8_t ds_smem[];
  uint8_t* ring = ds_smem;  // [DS_STAGES][32 K rows | 32 V rows]
  float* qs = reinterpret_cast<float*>(ring + DS_STAGES * C::STAGE);  // [2][NQ][D]
  uint64_t* full = reinterpret_cast<uint64_t*>(qs + 2 * C::Q_FLOATS);
  uint64_t* empty = full + DS_STAGES;
  int* abort_flag = reinterpret_cast<int*>(empty + DS_STAGES);
  float* cm = reinterpret_cast<float*>(abort_flag + 4);  // [DS_WARPS] m of each warp
  float* cl = cm + DS_WARPS;                           // [DS_WARPS] l of each warp
  float* cz = cl + DS_WARPS;                           // [DS_WARPS][D] weighted z
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < DS_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // the merge kernel may be launched now: its CTAs wait in grid_dep_wait
  // until this grid has completed and its summaries are visible
  grid_dep_launch_dependents();
  const WaitCtl w{nullptr, abort_flag, P.limit_ns};
  // this CTA's groups (an equal share of all keys, whatever the lengths)
  const int g_begin = (int)((long long)blockIdx.x * P.nitems / gridDim.x);
  const int g_end = (int)((long long)(blockIdx.x + 1) * P.nitems / gridDim.x);
  const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(P.K);
  const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(P.V);

  if (warp == DS_WARPS) {
    if (lane == 0) {
      // producer: group n of this CTA's sequence goes to stage n % DS_STAGES
      uint32_t n = 0;
      bool ok = true;
      int g = g_begin;
      DsPiece pc;
      while (ok && ds_next_piece(P, g, g_end, pc)) {
        const int k0 = pc.k0, k1 = pc.k1;
        const long long row0 = ((long long)pc.b * P.h + pc.head) * P.n_k;
        for (int k = k0; k < k1; k += 32, ++n) {
          const int s = n % DS_STAGES;
          if (n >= (uint32_t)DS_STAGES &&
              !mbar_wait(&empty[s], ((n / DS_STAGES) - 1) & 1, w)) {
            ok = false;
            break;
          }
          const uint32_t bytes = (uint32_t)min(32, k1 - k) * C::ROW;
          uint8_t* dst = ring + s * C::STAGE;
          mbar_arrive_expect_tx(&full[s], 2 * bytes);
          bulk_copy_g2s(dst, Kg + (row0 + k) * D, bytes, &full[s]);
          bulk_copy_g2s(dst + 32 * C::ROW, Vg + (row0 + k) * D, bytes, &full[s]);
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA exits
        for (uint32_t k = (n > (uint32_t)DS_STAGES ? n - DS_STAGES : 0); k < n; ++k)
          ds_drain(&full[k % DS_STAGES], (k / DS_STAGES) & 1);
      }
    }
  } else {
    const float cl2 = P.cl2;
    uint32_t n = 0;
    bool ok = true;
    int ik = 0;  // pieces of this CTA so far
    int g = g_begin;
    DsPiece pc;
    for (; ds_next_piece(P, g, g_end, pc); ++ik) {
      const int L = P.valid_len[pc.b];
      const int k0 = pc.k0, k1 = pc.k1;
      const long long bh = (long long)pc.b * P.h + pc.head;
      // the item's query rows, pre-multiplied by c log2(e), shared by the
      // consumer warps (double-buffered: a warp can only get here once every
      // warp has passed the previous item's barrier, i.e. has finished the
      // item before that, the last user of this buffer)
      float* q = qs + (ik & 1) * C::Q_FLOATS;
      const __nv_bfloat16* Qg = static_cast<const __nv_bfloat16*>(P.Q) + bh * P.n_q * D;
      for (int e = threadIdx.x; e < C::Q_FLOATS; e += 32 * DS_WARPS)
        q[e] = e < P.n_q * D ? __bfloat162float(Qg[e]) * cl2 : 0.f;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * DS_WARPS) : "memory");
      float m_run[NQ], l_run[NQ], z_run[NQ][CPL];
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        m_run[r] = -INFINITY;
        l_run[r] = 0.f;
#pragma unroll
        for (int t = 0; t < CPL; ++t) z_run[r][t] = 0.f;
      }
      for (int k = k0; k < k1; k += 32, ++n) {
        if ((int)(n % DS_WARPS) != warp) continue;
        const int s = n % DS_STAGES;
        // Stages are shared between consumer warps (DS_STAGES is not a
        // multiple of DS_WARPS): before waiting for group n's phase of the
        // stage, wait until group n - DS_STAGES (another warp's) has released
        // it, so that the stage's barrier is never two phases behind the
        // phase waited for (a parity wait cannot tell those apart). Group
        // n - 2 DS_STAGES is this warp's own, so the release barrier is never
        // two phases behind either.
        if (ok && n >= (uint32_t)DS_STAGES &&
            !mbar_wait(&empty[s], ((n / DS_STAGES) - 1) & 1, w))
          ok = false;
        if (ok && !mbar_wait(&full[s], (n / DS_STAGES) & 1, w)) ok = false;
        if (!__all_sync(0xffffffffu, ok)) {  // gave up: keep to the item loop, do no work
          ok = false;
          continue;
        }
        const int rows = min(32, k1 - k);
        const uint8_t* kst = ring + s * C::STAGE;
        const uint8_t* vst = kst + 32 * C::ROW;
        // scores of this lane's key (row `lane` of the group) against every
        // query row; lane j starts at 16-byte chunk j of its row, so the 32
        // lanes' reads spread over the shared-memory banks
        float sc[NQ];
#pragma unroll
        for (int r = 0; r < NQ; ++r) sc[r] = 0.f;
        if (lane < rows) {
          const uint8_t* krow = kst + lane * C::ROW;
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            const int c = (i + lane) & (NCH - 1);
            float kv[8];
            Vec16<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(krow + c * 16), kv);
#pragma unroll
            for (int r = 0; r < NQ; ++r) {
              const float4 q0 = *reinterpret_cast<const float4*>(q + r * D + c * 8);
              const float4 q1 = *reinterpret_cast<const float4*>(q + r * D + c * 8 + 4);
              float acc = sc[r];
              acc = fmaf(q0.x, kv[0], acc);
              acc = fmaf(q0.y, kv[1], acc);
              acc = fmaf(q0.z, kv[2], acc);
              acc = fmaf(q0.w, kv[3], acc);
              acc = fmaf(q1.x, kv[4], acc);
              acc = fmaf(q1.y, kv[5], acc);
              acc = fmaf(q1.z, kv[6], acc);
              acc = fmaf(q1.w, kv[7], acc);
              sc[r] = acc;
            }
          }
        }
        // fold the group into each row's summary (base 2)
        const int key = k + lane;
        float p[NQ];
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
          p[r] = 0.f;
          if (r >= P.n_q) continue;  // uniform
          bool allowed = lane < rows;
          if (P.causal_tail) allowed = allowed && key <= L - P.n_q + r;
          const float sv = allowed ? sc[r] : -INFINITY;
          const float m_blk = dwarp_max(sv);
          if (m_blk == -INFINITY) continue;  // the empty summary
          const float m_new = fmaxf(m_run[r], m_blk);
          const float a = exp2f(m_run[r] - m_new);
          p[r] = allowed ? exp2f(sv - m_new) : 0.f;
          l_run[r] = l_run[r] * a + dwarp_sum(p[r]);
#pragma unroll
          for (int t = 0; t < CPL; ++t) z_run[r][t] *= a;
          m_run[r] = m_new;
        }
        // z += sum over the group's keys of p_j v_j; lane owns CPL columns
        for (int j = 0; j < rows; ++j) {
          float vv[CPL];
          const uint8_t* vp = vst + j * C::ROW + lane * CPL * 2;
          if constexpr (CPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(vp);
            vv[0] = __uint_as_float(u.x << 16);
            vv[1] = __uint_as_float(u.x & 0xffff0000u);
            vv[2] = __uint_as_float(u.y << 16);
            vv[3] = __uint_as_float(u.y & 0xffff0000u);
          } else {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(vp);
            vv[0] = __uint_as_float(u << 16);
            vv[1] = __uint_as_float(u & 0xffff0000u);
          }
#pragma unroll
          for (int r = 0; r < NQ; ++r) {
            const float pj = __shfl_sync(0xffffffffu, p[r], j);
#pragma unroll
            for (int t = 0; t < CPL; ++t) z_run[r][t] = fmaf(pj, vv[t], z_run[r][t]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled
      }
      // The piece's summary of each row: the merge of the warps' summaries
      // (those that took no group are empty), combined through shared
      // memory, into the piece's slot of the row.
#pragma unroll 1
      for (int r = 0; r < P.n_q && r < NQ; ++r) {
        constexpr int NT = 32 * DS_WARPS;
        float mr = m_run[0], lr = l_run[0];
#pragma unroll
        for (int rr = 1; rr < NQ; ++rr)
          if (rr == r) {
            mr = m_run[rr];
            lr = l_run[rr];
          }
        if (lane == 0) {
          cm[warp] = mr;
          cl[warp] = lr;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
        float M = cm[0];
#pragma unroll
        for (int i = 1; i < DS_WARPS; ++i) M = fmaxf(M, cm[i]);
        const float wgt = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
#pragma unroll
        for (int rr = 0; rr < NQ; ++rr)
          if (rr == r) {
#pragma unroll
            for (int t = 0; t < CPL; ++t) cz[warp * D + lane * CPL + t] = z_run[rr][t] * wgt;
          }
        asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
        float* dst = P.part + ((bh * P.n_q + r) * P.nsplit + pc.slot) * (long long)(2 + D);
        for (int c = threadIdx.x; c < D; c += NT) {
          float zc = 0.f;
#pragma unroll
          for (int i = 0; i < DS_WARPS; ++i) zc += cz[i * D + c];
          dst[2 + c] = zc;
          if (pc.clear_rest) dst[(2 + D) + 2 + c] = 0.f;  // the chunk's second slot: empty
        }
        if (pc.clear_rest && threadIdx.x == 0) {
          dst[(2 + D)] = -INFINITY;
          dst[(2 + D) + 1] = 0.f;
        }
        if (threadIdx.x == 0) {
          float l = 0.f;
#pragma unroll
          for (int i = 0; i < DS_WARPS; ++i)
            if (cm[i] != -INFINITY) l += exp2f(cm[i] - M) * cl[i];
          dst[0] = M;
          dst[1] = l;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");  // cm, cl, cz free again
      }
    }
  }
}

// Pass 2. grid (n_q, h, B), 256 threads: merges the splits of one query row
// (those below the valid length) and writes z / l.
template <typename T>
__global__ void __launch_bounds__(DEC_THREADS) decode_merge_kernel(
    const __grid_constant__ DecodeParams P) {
  __shared__ float w[1024];
  __shared__ float red[DEC_WARPS];
  __shared__ float bcast;
  // launched as a dependent of pass 1 (programmatic stream serialization):
  // its summaries are complete and visible once this returns
  grid_dep_wait();
  const int row = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  const int L = P.valid_len[b];
  const int nsp = ((L + DEC_CHUNK - 1) / DEC_CHUNK) * P.per_chunk;
  const int dv = P.d_vh;
  const long long bh = (long long)b * P.h + head;
  const float* src = P.part + (bh * P.n_q + row) * P.nsplit * (long long)(2 + dv);
  // M = max of the splits' m (empty splits have m = -inf)
  float mx = -INFINITY;
  for (int s = threadIdx.x; s < nsp; s += DEC_THREADS) mx = fmaxf(mx, src[(long long)s * (2 + dv)]);
  mx = dwarp_max(mx);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = red[0];
    for (int i = 1; i < DEC_WARPS; ++i) v = fmaxf(v, red[i]);
    bcast = v;
  }
  __syncthreads();
  const float M = bcast;
  // weights e^{m_s - M} (base 2) and l = sum_s l_s e^{m_s - M}
  float lsum = 0.f;
  for (int s = threadIdx.x; s < nsp; s += DEC_THREADS) {
    const float m = src[(long long)s * (2 + dv)];
    const float ws = (m == -INFINITY) ? 0.f : exp2f(m - M);
    w[s] = ws;
    lsum += ws * src[(long long)s * (2 + dv) + 1];
  }
  lsum = dwarp_sum(lsum);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = lsum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.f;
    for (int i = 0; i < DEC_WARPS; ++i) v += red[i];
    bcast = v;
  }
  __syncthreads();
  const float inv = 1.f / bcast;
  T* zrow = static_cast<T*>(P.Z) + ((long long)b * P.n_q + row) * (long long)P.h * dv +
            (long long)head * dv;
  // z = sum_s w_s z_s, every thread busy: G groups of dv threads, group g
  // summing the splits s = g, g + G, ..., eight loads in flight per thread;
  // the groups' sums are then added through shared memory
  __shared__ float zpart[DEC_THREADS];
  const int G = DEC_THREADS / dv;  // d_vh <= 256: at least 1
  const int col = threadIdx.x % dv, grp = threadIdx.x / dv;
  float z = 0.f;
  if (grp < G) {
    float za[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int s = grp;
    for (; s + 7 * G < nsp; s += 8 * G) {
#pragma unroll
      for (int u = 0; u < 8; ++u)
        za[u] = fmaf(w[s + u * G], src[(long long)(s + u * G) * (2 + dv) + 2 + col], za[u]);
    }
    for (; s < nsp; s += G) za[0] = fmaf(w[s], src[(long long)s * (2 + dv) + 2 + col], za[0]);
    z = ((za[0] + za[1]) + (za[2] + za[3])) + ((za[4] + za[5]) + (za[6] + za[7]));
  }
  zpart[threadIdx.x] = z;
  __syncthreads();
  if (threadIdx.x < dv) {
    float t = 0.f;
    for (int g = 0; g < G; ++g) t += zpart[g * dv + threadIdx.x];
    if (sizeof(T) == 4)
      reinterpret_cast<float*>(zrow)[threadIdx.x] = t * inv;
    else
      reinterpret_cast<__nv_bfloat16*>(zrow)[threadIdx.x] = __float2bfloat16_rn(t * inv);
  }
}

template <typename T, int DQK, int DV>
bool launch_fast(const DecodeParams& P, const dim3& g1, cudaStream_t s) {
  if (P.d_h != DQK || P.d_vh != DV) return false;
  if (P.n_q == 1)
    decode_partial_fast_kernel<T, 1, DQK, DV><<<g1, DEC_THREADS, 0, s>>>(P);
  else if (P.n_q == 2)
    decode_partial_fast_kernel<T, 2, DQK, DV><<<g1, DEC_THREADS, 0, s>>>(P);
  else if (P.n_q <= 4)
    decode_partial_fast_kernel<T, 4, DQK, DV><<<g1, DEC_THREADS, 0, s>>>(P);
  else
    decode_partial_fast_kernel<T, 8, DQK, DV><<<g1, DEC_THREADS, 0, s>>>(P);
  return true;
}

template <int NQ, int D>
bool launch_stream(const DecodeParams& P, cudaStream_t s) {
  using C = DsCfg<NQ, D>;
  if (!ensure_smem_limit((const void*)decode_stream_kernel<NQ, D>, C::SMEM)) return false;
  // as many CTAs as can be resident at once (shared memory and registers),
  // asked once per device
  const int per_sm = resident_ctas((const void*)decode_stream_kernel<NQ, D>, DS_THREADS, C::SMEM);
  const int cap = num_sms() * per_sm;
  // at least a chunk's worth of groups per CTA (so a chunk has at most two
  // pieces)
  const int want = P.nitems / DS_CHUNK_GROUPS;
  const int grid = want < 1 ? 1 : (want < cap ? want : cap);
  decode_stream_kernel<NQ, D><<<grid, DS_THREADS, C::SMEM, s>>>(P);
  return true;
}

template <int D>
bool launch_stream_rows(const DecodeParams& P, cudaStream_t s) {
  if (P.n_q == 1) return launch_stream<1, D>(P, s);
  if (P.n_q == 2) return launch_stream<2, D>(P, s);
  if (P.n_q <= 4) return launch_stream<4, D>(P, s);
  return launch_stream<8, D>(P, s);
}

template <typename T>
mha_status launch_decode(DecodeParams& P, int nchunk, cudaStream_t s) {
  const dim3 g1(nchunk, P.h, P.B), g2(P.n_q, P.h, P.B);
  if (sizeof(T) == 2 && P.d_h == P.d_vh && (P.d_h == 64 || P.d_h == 128) && P.n_q <= 8) {
    // streaming pass 1: the 32-key groups of every (batch item, head)
    // sequence, batch item by batch item, shared out in equal ranges
    long long groups = 0;
    for (int b = 0; b < P.B; ++b) {
      P.item_start[b] = (int)groups;
      groups += (long long)P.h * ((P.valid_len[b] + DS_GROUP - 1) / DS_GROUP);
    }
    if (groups < (1ll << 30)) {
      P.item_start[P.B] = (int)groups;
      P.nitems = (int)groups;
      P.per_chunk = 2;  // two summary slots per chunk (a range boundary may cut it)
      const bool ok = P.d_h == 64 ? launch_stream_rows<64>(P, s) : launch_stream_rows<128>(P, s);
      if (!ok) return MHA_ERR_CUDA;
      // the merge follows pass 1 without a launch gap
      const cudaError_t e = launch_dependent(decode_merge_kernel<T>, g2, dim3(DEC_THREADS), 0, s, P);
      count_launch(2);
      return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
    }
  }
  if (launch_fast<T, 64, 64>(P, g1, s) || launch_fast<T, 128, 128>(P, g1, s)) {
    decode_merge_kernel<T><<<g2, DEC_THREADS, 0, s>>>(P);
    count_launch(2);
    return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
  }
  const bool vec = P.d_h % 8 == 0;
  if (P.d_vh <= 64) {
    if (vec) decode_partial_kernel<T, 2, true><<<g1, DEC_THREADS, 0, s>>>(P);
    else decode_partial_kernel<T, 2, false><<<g1, DEC_THREADS, 0, s>>>(P);
  } else if (P.d_vh <= 128) {
    if (vec) decode_partial_kernel<T, 4, true><<<g1, DEC_THREADS, 0, s>>>(P);
    else decode_partial_kernel<T, 4, false><<<g1, DEC_THREADS, 0, s>>>(P);
  } else {
    if (vec) decode_partial_kernel<T, 8, true><<<g1, DEC_THREADS, 0, s>>>(P);
    else decode_partial_kernel<T, 8, false><<<g1, DEC_THREADS, 0, s>>>(P);
  }
  decode_merge_kernel<T><<<g2, DEC_THREADS, 0, s>>>(P);
  count_launch(2);
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace

size_t decode_workspace_bytes(int B, int n_q, int n_k, int h, int d_vh) {
  const size_t nsplit = (size_t)((n_k + DEC_CHUNK - 1) / DEC_CHUNK) * DEC_WARPS;
  return (size_t)B * h * n_q * nsplit * (2 + (size_t)d_vh) * sizeof(float);
}

mha_status attention_decode(const DecodeArgs& a, mha_dtype dt, cudaStream_t s) {
  if (a.d_h > 256 || a.d_vh > 256) return MHA_ERR_UNSUPPORTED;
  const int nchunk = (a.n_k + DEC_CHUNK - 1) / DEC_CHUNK;
  if (nchunk * DEC_WARPS > 1024) return MHA_ERR_UNSUPPORTED;  // merge weights in shared memory
  if (a.h > 65535 || a.B > 65535) return MHA_ERR_UNSUPPORTED;
  DecodeParams P;
  P.Q = a.Q;
  P.K = a.K;
  P.V = a.V;
  P.Z = a.Z;
  P.part = static_cast<float*>(a.part);
  P.B = a.B;
  P.n_q = a.n_q;
  P.n_k = a.n_k;
  P.h = a.h;
  P.d_h = a.d_h;
  P.d_vh = a.d_vh;
  P.nsplit = nchunk * DEC_WARPS;
  P.per_chunk = DEC_WARPS;
  P.cl2 = a.c * 1.4426950408889634f;
  P.causal_tail = a.causal_tail;
  P.limit_ns = wait_limit_ns();
  P.nitems = 0;
  for (int b = 0; b < MHA_MAX_PADDED_BATCH; ++b)
    P.valid_len[b] = (a.cache_len_host && b < a.B) ? a.cache_len_host[b] : a.n_k;
  if (dt == MHA_DTYPE_F32) return launch_decode<float>(P, nchunk, s);
  return launch_decode<__nv_bfloat16>(P, nchunk, s);
}

}  // namespace mha
