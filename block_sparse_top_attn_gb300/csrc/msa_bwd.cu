// MSA block-sparse attention backward on sm_103a: preprocess, main KV-parallel
// tcgen05 kernel and postprocess ("msa_backward_sm100" page: KV-parallel task
// rows of 8 queries x 16 heads bucketed by (batch, index head, key block); five
// GEMMs S, dP, dV, dK, dQ; dK/dV accumulated per bucket segment; dQ reduced
// into an accumulator that the postprocess casts to bf16).
//
// Main kernel data flow for one task (128 rows = 8 tokens x 16 q-heads, one
// key block of 64 keys, head_dim 128), all GEMMs M = 128 with fp32 in TMEM:
//   S    [row, key] = Q  . K^T          A = Q  (K-major)  B = K  (K-major)
//   dP   [row, key] = dO . V^T          A = dO (K-major)  B = V  (K-major)
//   P  = exp2(S * scale * log2e - LSE * log2e) on the causal mask, else 0
//   dS = scale * P * (dP - D)           (both rounded to bf16 in smem)
//   dV^T [d, key] += dO^T . P           A = dO (MN-major) B = P  (MN-major)
//   dK^T [d, key] += Q^T  . dS          A = Q  (MN-major) B = dS (MN-major)
//   dQ   [row, d]  = dS . K             A = dS (K-major)  B = K  (MN-major)
// Q, dO, K, V arrive by TMA with 128-byte swizzle; P and dS are written in the
// same swizzled layout, so no operand is ever transposed in memory.  dQ is
// reduced into an fp32 accumulator with TMA bulk reduce-add per task; dK^T and
// dV^T stay in TMEM for a bucket segment and are reduced the same way when the
// segment ends.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa_common.cuh"
#include "msa_host.cuh"
#include "msa_tmap.cuh"

namespace msa {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// preprocess: D[t, h] = sum_d dO * O (fp32) and zeroed fp32 accumulators
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                          float* __restrict__ delta, int64_t rows,
                                                          float4* __restrict__ zero, int64_t zero_n4,
                                                          const int32_t* status) {
  if (status_bad(status)) return;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  // 16 threads per row of 128 bf16 (16 bytes each)
  const int64_t total16 = rows * 16;
  for (int64_t i = tid; i < (total16 + 31) / 32 * 32; i += nthr) {
    float acc = 0.f;
    if (i < total16) {
      const uint4 a = o[i], b = dout[i];
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc += __uint_as_float(av[j] << 16) * __uint_as_float(bv[j] << 16);
        acc += __uint_as_float(av[j] & 0xFFFF0000u) * __uint_as_float(bv[j] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (i < total16 && (i & 15) == 0) delta[i >> 4] = acc;
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = tid; i < zero_n4; i += nthr) zero[i] = z;
}

// ---------------------------------------------------------------------------
// postprocess: bf16 casts; K/V rows outside every document are written as 0
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 cast8(const float4* src) {
  const float4 a = src[0], b = src[1];
  return make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
}

__global__ void __launch_bounds__(256) postprocess_kernel(const float4* __restrict__ dq_acc, uint4* __restrict__ dq,
                                                           int64_t dq_n8, const float4* __restrict__ dk_acc,
                                                           const float4* __restrict__ dv_acc, uint4* __restrict__ dk,
                                                           uint4* __restrict__ dv, int64_t kv_n8, int kv_row_n8,
                                                           const int32_t* cu, const int32_t* kvs, int N,
                                                           const int32_t* status) {
  if (status_bad(status)) return;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = tid; i < dq_n8; i += nthr) dq[i] = cast8(dq_acc + 2 * i);
  for (int64_t i = tid; i < kv_n8; i += nthr) {
    const int64_t row = i / kv_row_n8;
    int lo = 0, hi = N - 1;  // last document starting at or before row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (kvs[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const bool inside = row >= kvs[lo] && row < (int64_t)kvs[lo] + (cu[lo + 1] - cu[lo]);
    if (inside) {
      dk[i] = cast8(dk_acc + 2 * i);
      dv[i] = cast8(dv_acc + 2 * i);
    } else {
      dk[i] = make_uint4(0, 0, 0, 0);
      dv[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// main kernel, synchronous form: one thread issues TMA and MMA, 4 warps own the
// 128 TMEM lanes for the softmax / dS math and the flushes.
// ---------------------------------------------------------------------------
struct MainArgs {
  const float* lse;
  const float* delta;
  const int32_t* meta;
  const int32_t* q_rows;
  const int32_t* q_pos;
  const int32_t* walk;
  const int32_t* kv_doc_starts;
  int Hq;
  float scale_log2;
  float scale;
  int32_t* status;
};

namespace v0 {
constexpr uint32_t OFF_Q = 0;           // [2 halves][128 rows][128 B]
constexpr uint32_t OFF_DO = 32768;
constexpr uint32_t OFF_K = 65536;       // [2 halves][64 keys][128 B]
constexpr uint32_t OFF_V = 81920;
constexpr uint32_t OFF_P = 98304;       // [128 rows][64 keys bf16]
constexpr uint32_t OFF_DS = 114688;
constexpr uint32_t OFF_ST = 131072;     // 64 KB fp32 staging for TMA reduce-add
constexpr uint32_t OFF_BAR = 196608;
constexpr uint32_t SMEM = OFF_BAR + 64 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_DP = 64, COL_DQ = 128, COL_DK = 256, COL_DV = 320;
}  // namespace v0

// Write dK^T / dV^T (TMEM lane = d, column = key) as fp32 [64 keys][32 d]
// swizzled quarters and reduce-add them into the fp32 accumulators.
__device__ __forceinline__ void flush_dkdv_v0(uint8_t* sm, uint32_t tmem, const CUtensorMap* tmdK,
                                              const CUtensorMap* tmdV, int hi, int kvrow) {
  using namespace v0;
  const int tid = threadIdx.x, warp = tid >> 5, dd = tid & 31;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (tid == 0) bulk_wait_read_all();
  __syncthreads();
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint32_t col = which == 0 ? COL_DK : COL_DV;
    uint8_t* qbuf = sm + OFF_ST + which * 32768 + warp * 8192;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + lane_base + col + c0, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int key = c0 + j;
        *reinterpret_cast<uint32_t*>(qbuf + key * 128 + ((((dd >> 2) ^ (key & 7))) << 4) + (dd & 3) * 4) = v[j];
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    for (int qq = 0; qq < 4; ++qq) {
      tma_reduce_add_3d(tmdK, sm + OFF_ST + qq * 8192, qq * 32, hi, kvrow);
      tma_reduce_add_3d(tmdV, sm + OFF_ST + 32768 + qq * 8192, qq * 32, hi, kvrow);
    }
    bulk_commit();
  }
}

__global__ void __launch_bounds__(128, 1)
    bwd_main_v0(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
                const __grid_constant__ CUtensorMap tmdV, MainArgs a) {
  using namespace v0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_load + 2);
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t sbase = smem_u32(sm);

  constexpr uint32_t ID_S = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t ID_T = idesc_bf16_f32(128, 64, true, true);
  constexpr uint32_t ID_Q = idesc_bf16_f32(128, 128, false, true);

  uint32_t ph_load = 0, ph_mma = 0;
  bool aborted = status_bad(a.status);
  const int n = a.walk[MSA_WALK_ROWS], R = a.walk[MSA_WALK_ROWS_PER_CTA];
  const int full = a.walk[MSA_WALK_FULL], grid = a.walk[MSA_WALK_GRID];

  for (int u = blockIdx.x; u < grid && !aborted; u += gridDim.x) {
    int t0, step, cnt;
    if (u < full) {
      t0 = u * R; step = 1; cnt = R;
    } else {
      step = grid - full; t0 = full * R + (u - full); cnt = (n - t0 + step - 1) / step;
    }
    int cur_hi = -1, cur_r = -1, kvrow = 0;
    bool seg_active = false, seg_first = true;
    for (int i = 0; i < cnt && !aborted; ++i) {
      const int t = t0 + i * step;
      const int* mt = a.meta + (int64_t)t * MSA_TASK_META_COLS;
      const int hi = mt[0], r = mt[1], d = mt[4], b = mt[5];
      const bool new_bucket = hi != cur_hi || r != cur_r;
      if (new_bucket && seg_active) {
        flush_dkdv_v0(sm, tmem, &tmdK, &tmdV, cur_hi, kvrow);
        seg_active = false;
      }
      const int tok0 = a.q_rows[(int64_t)t * 8];
      if (new_bucket) {
        cur_hi = hi; cur_r = r; kvrow = a.kv_doc_starts[d] + b * 64; seg_first = true;
      }
      if (tid == 0) {
        mbar_arrive_expect_tx(bar_load, 65536u + (new_bucket ? 32768u : 0u));
        tma_load_3d(sm + OFF_Q, &tmQ, bar_load, 0, hi * 16, tok0);
        tma_load_3d(sm + OFF_Q + 16384, &tmQ, bar_load, 64, hi * 16, tok0);
        tma_load_3d(sm + OFF_DO, &tmdO, bar_load, 0, hi * 16, tok0);
        tma_load_3d(sm + OFF_DO + 16384, &tmdO, bar_load, 64, hi * 16, tok0);
        if (new_bucket) {
          tma_load_3d(sm + OFF_K, &tmK, bar_load, 0, hi, kvrow);
          tma_load_3d(sm + OFF_K + 8192, &tmK, bar_load, 64, hi, kvrow);
          tma_load_3d(sm + OFF_V, &tmV, bar_load, 0, hi, kvrow);
          tma_load_3d(sm + OFF_V + 8192, &tmV, bar_load, 64, hi, kvrow);
        }
      }
      if (!mbar_wait(bar_load, ph_load, a.status)) aborted = true;
      ph_load ^= 1;
      if (__syncthreads_or(aborted)) { aborted = true; break; }

      // S = Q K^T, dP = dO V^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
          umma_bf16(tmem + COL_S, sdesc_sw128(sbase + OFF_Q + half * 16384 + sub, 16, 1024),
                    sdesc_sw128(sbase + OFF_K + half * 8192 + sub, 16, 1024), ID_S, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
          umma_bf16(tmem + COL_DP, sdesc_sw128(sbase + OFF_DO + half * 16384 + sub, 16, 1024),
                    sdesc_sw128(sbase + OFF_V + half * 8192 + sub, 16, 1024), ID_S, kk > 0);
        }
        umma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, ph_mma, a.status)) aborted = true;
      ph_mma ^= 1;
      if (__syncthreads_or(aborted)) { aborted = true; break; }
      tc_fence_after();

      // P and dS for row tid (token slot tid / 16, head tid % 16)
      {
        const int slot = tid >> 4, hh = tid & 15;
        const int qpos = a.q_pos[(int64_t)t * 8 + slot];
        float lse2 = 0.f, dlt = 0.f;
        if (qpos >= 0) {
          const int64_t row = (int64_t)(tok0 + slot) * a.Hq + hi * 16 + hh;
          lse2 = a.lse[row] * kLog2e;
          dlt = a.delta[row];
        }
        const int kbase = b * 64;
        uint32_t pk[32], dk[32];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t sv[16], dpv[16];
          tmem_ld16(tmem + lane_base + COL_S + c0, sv);
          tmem_ld16(tmem + lane_base + COL_DP + c0, dpv);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float p[2], ds[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const bool valid = qpos >= 0 && kbase + c0 + j + e <= qpos;
              const float pv = ex2_approx(__uint_as_float(sv[j + e]) * a.scale_log2 - lse2);
              p[e] = valid ? pv : 0.f;
              ds[e] = valid ? pv * (__uint_as_float(dpv[j + e]) - dlt) * a.scale : 0.f;
            }
            pk[(c0 + j) >> 1] = pack_bf16x2(p[0], p[1]);
            dk[(c0 + j) >> 1] = pack_bf16x2(ds[0], ds[1]);
          }
        }
        uint8_t* prow = sm + OFF_P + tid * 128;
        uint8_t* drow = sm + OFF_DS + tid * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t o = (uint32_t)((c ^ (tid & 7)) << 4);
          *reinterpret_cast<uint4*>(prow + o) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          *reinterpret_cast<uint4*>(drow + o) = make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();

      // dV^T += dO^T P, dK^T += Q^T dS, dQ = dS K
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          umma_bf16(tmem + COL_DV, sdesc_sw128(sbase + OFF_DO + kk * 2048, 16384, 1024),
                    sdesc_sw128(sbase + OFF_P + kk * 2048, 8192, 1024), ID_T, (kk > 0 || !seg_first) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          umma_bf16(tmem + COL_DK, sdesc_sw128(sbase + OFF_Q + kk * 2048, 16384, 1024),
                    sdesc_sw128(sbase + OFF_DS + kk * 2048, 8192, 1024), ID_T, (kk > 0 || !seg_first) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          umma_bf16(tmem + COL_DQ, sdesc_sw128(sbase + OFF_DS + kk * 32, 16, 1024),
                    sdesc_sw128(sbase + OFF_K + kk * 2048, 8192, 1024), ID_Q, kk > 0);
        }
        umma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, ph_mma, a.status)) aborted = true;
      ph_mma ^= 1;
      if (__syncthreads_or(aborted)) { aborted = true; break; }
      tc_fence_after();
      seg_first = false;
      seg_active = true;

      // dQ: TMEM -> swizzled fp32 staging -> TMA reduce-add into the accumulator
      if (tid == 0) bulk_wait_read_all();
      __syncthreads();
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t v[32];
        tmem_ld16(tmem + lane_base + COL_DQ + qq * 32, *reinterpret_cast<uint32_t(*)[16]>(v));
        tmem_ld16(tmem + lane_base + COL_DQ + qq * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        tmem_ld_wait();
        uint8_t* row = sm + OFF_ST + qq * 16384 + tid * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(row + ((c ^ (tid & 7)) << 4)) =
              make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        for (int qq = 0; qq < 4; ++qq) tma_reduce_add_3d(&tmdQ, sm + OFF_ST + qq * 16384, qq * 32, hi * 16, tok0);
        bulk_commit();
      }
    }
    if (seg_active && !aborted) flush_dkdv_v0(sm, tmem, &tmdK, &tmdV, cur_hi, kvrow);
  }
  if (tid == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace msa

#include "msa_bwd_ws.cuh"

using namespace msa;

extern "C" int msa_bwd_staged(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                              const uint16_t* o, const uint16_t* dout, const float* lse, const int32_t* task_meta,
                              const int32_t* task_q_rows, const int32_t* task_q_pos, const int32_t* walk,
                              int64_t task_cap, uint16_t* dq, uint16_t* dk, uint16_t* dv, int32_t* d_status,
                              void* ws, size_t ws_bytes, void* stream, uint32_t stages) {
  int rc = check_problem(p);
  if (rc) return rc;
  const void* ptrs[] = {q, k, v, o, dout, lse, task_meta, task_q_rows, task_q_pos, walk, dq, dk, dv, d_status, ws};
  for (const void* x : ptrs)
    if (!x || !aligned16(x)) return MSA_ERR_INVALID_ARGUMENT;
  if (task_cap < 1 || task_cap > INT32_MAX) return MSA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < bwd_ws_bytes(p)) return MSA_ERR_INVALID_ARGUMENT;
  if ((rc = check_device_current())) return rc;
  int32_t sms = 0;
  if ((rc = sm_count_current(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t T = p->total_tokens, Hq = p->num_q_heads, W = p->kv_rows, Hkv = p->num_kv_heads;

  uint8_t* w = static_cast<uint8_t*>(ws);
  float* delta = reinterpret_cast<float*>(w);
  w += round_up(sizeof(float) * T * Hq, 256);
  float* dq_acc = reinterpret_cast<float*>(w);
  w += round_up(sizeof(float) * T * Hq * kHeadDim, 256);
  float* dk_acc = reinterpret_cast<float*>(w);
  w += round_up(sizeof(float) * W * Hkv * kHeadDim, 256);
  float* dv_acc = reinterpret_cast<float*>(w);
  w += round_up(sizeof(float) * W * Hkv * kHeadDim, 256);
  const int64_t zero_n4 = (reinterpret_cast<float*>(w) - dq_acc) / 4;

  // loads: Q/dO boxes of 8 tokens x 16 heads x 64 dims, K/V boxes of 64 keys x 64 dims;
  // reduce-adds: dQ boxes of 2 tokens x 16 heads x 32 dims, dK/dV of 32 keys x 32 dims (fp32)
  CUtensorMap tmQ, tmdO, tmK, tmV, tmdQ, tmdK, tmdV;
  bool ok = make_tmap_3d(&tmQ, q, false, T, Hq, 64, 16, 8) && make_tmap_3d(&tmdO, dout, false, T, Hq, 64, 16, 8) &&
            make_tmap_3d(&tmK, k, false, W, Hkv, 64, 1, 64) && make_tmap_3d(&tmV, v, false, W, Hkv, 64, 1, 64) &&
            make_tmap_3d(&tmdQ, dq_acc, true, T, Hq, 32, 16, 2) &&
            make_tmap_3d(&tmdK, dk_acc, true, W, Hkv, 32, 1, 32) &&
            make_tmap_3d(&tmdV, dv_acc, true, W, Hkv, 32, 1, 32);
  if (!ok) return MSA_ERR_CUDA;

  if (stages & ~(uint32_t)MSA_STAGE_ALL) return MSA_ERR_INVALID_ARGUMENT;
  if (stages & MSA_STAGE_PREPROCESS)
    preprocess_kernel<<<sms * 8, 256, 0, st>>>(reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout),
                                             delta, T * Hq, reinterpret_cast<float4*>(dq_acc), zero_n4, d_status);
  if (stages & MSA_STAGE_MAIN) {
  if (cudaFuncSetAttribute(bwd_main_ws, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ws::SMEM) != cudaSuccess)
    return MSA_ERR_CUDA;
  const int64_t bound = msa_grid_launch_bound(task_cap, sms);
  const int grid = (int)(bound < sms ? (bound < 1 ? 1 : bound) : sms);
  MainArgs a;
  a.lse = lse; a.delta = delta; a.meta = task_meta; a.q_rows = task_q_rows; a.q_pos = task_q_pos; a.walk = walk;
  a.kv_doc_starts = p->kv_doc_starts; a.Hq = (int)Hq; a.scale_log2 = p->softmax_scale * kLog2e;
  a.scale = p->softmax_scale; a.status = d_status;
  bwd_main_ws<<<grid, ws::kThreads, ws::SMEM, st>>>(tmQ, tmdO, tmK, tmV, tmdQ, tmdK, tmdV, a);
  }
  if (stages & MSA_STAGE_POSTPROCESS)
    postprocess_kernel<<<sms * 8, 256, 0, st>>>(
      reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint4*>(dq), T * Hq * kHeadDim / 8,
      reinterpret_cast<const float4*>(dk_acc), reinterpret_cast<const float4*>(dv_acc), reinterpret_cast<uint4*>(dk),
      reinterpret_cast<uint4*>(dv), W * Hkv * kHeadDim / 8, (int)(Hkv * kHeadDim / 8), p->cu_seqlens,
      p->kv_doc_starts, p->num_docs, d_status);
  return cuda_status(cudaGetLastError());
}

extern "C" int msa_bwd(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const uint16_t* o, const uint16_t* dout, const float* lse, const int32_t* task_meta,
                       const int32_t* task_q_rows, const int32_t* task_q_pos, const int32_t* walk,
                       int64_t task_cap, uint16_t* dq, uint16_t* dk, uint16_t* dv, int32_t* d_status, void* ws,
                       size_t ws_bytes, void* stream) {
  return msa_bwd_staged(p, q, k, v, o, dout, lse, task_meta, task_q_rows, task_q_pos, walk, task_cap, dq, dk, dv,
                        d_status, ws, ws_bytes, stream, MSA_STAGE_ALL);
}
