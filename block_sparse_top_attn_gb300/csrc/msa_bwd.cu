// MSA block-sparse attention backward on sm_103a: preprocess, main KV-parallel
// tcgen05 kernel and postprocess ("msa_backward_sm100" page: KV-parallel task
// rows of 8 queries x 16 heads bucketed by (batch, index head, key block); five
// GEMMs S, dP, dV, dK, dQ; dK/dV accumulated per bucket segment; dQ reduced
// in bf16 across tasks, as the pages' bf16 dQ pool is).
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
// same swizzled layout, so no operand is ever transposed in memory.  A task's
// dQ (fp32 in TMEM over its 64 keys) is rounded to bf16 and reduced straight
// into the bf16 dQ output with a TMA bulk reduce-add (or, with the fp32 dQ
// option, reduce-added in fp32 into a workspace accumulator that the
// postprocess rounds once); dK^T and dV^T stay in
// TMEM for a bucket segment and are reduced into fp32 accumulators when the
// segment ends, which the postprocess casts to bf16.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa_common.cuh"
#include "msa_host.cuh"
#include "msa_tmap.cuh"

namespace msa {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// preprocess: D[t, h] = sum_d dO * O (fp32), zeroed dK/dV fp32 accumulators and
// bf16 dQ output
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                          float* __restrict__ delta, int64_t T, int Hq,
                                                          float4* __restrict__ zero,
                                                          int64_t zero_n4, uint4* __restrict__ dq_zero,
                                                          int64_t dq_zero_n16, const int32_t* status) {
  if (status_bad(status)) return;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  // 16 threads per row of 128 bf16 (16 bytes each)
  const int64_t total16 = T * Hq * 16;
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
  // the buffer dQ is reduced into: the bf16 output, or the fp32 accumulator
  const uint4 zb = make_uint4(0, 0, 0, 0);
  for (int64_t i = tid; i < dq_zero_n16; i += nthr) dq_zero[i] = zb;
}

// ---------------------------------------------------------------------------
// postprocess: bf16 casts; K/V rows outside every document are written as 0
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 cast8(const float4* src) {
  const float4 a = src[0], b = src[1];
  return make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
}

// The dK, dV accumulators are index-head-major, [Hkv][W][128]; the outputs are
// [W][Hkv][128].  dQ needs a cast only when it was accumulated in fp32
// (dq_acc non-null, same layout as the output); otherwise it was reduced
// straight into its bf16 output.
__global__ void __launch_bounds__(256) postprocess_kernel(const float4* __restrict__ dk_acc,
                                                           const float4* __restrict__ dv_acc, uint4* __restrict__ dk,
                                                           uint4* __restrict__ dv, int64_t kv_n8, int64_t W, int Hkv,
                                                           const int32_t* cu, const int32_t* kvs, int N,
                                                           const float4* __restrict__ dq_acc,
                                                           uint4* __restrict__ dq, int64_t dq_n8,
                                                           const int32_t* status) {
  if (status_bad(status)) return;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  if (dq_acc)
    for (int64_t i = tid; i < dq_n8; i += nthr) dq[i] = cast8(dq_acc + 2 * i);
  const int kv_row_n8 = Hkv * 16;
  for (int64_t i = tid; i < kv_n8; i += nthr) {
    const int64_t row = i / kv_row_n8;
    const int r = (int)(i - row * kv_row_n8);
    const int64_t src = ((int64_t)(r >> 4) * W + row) * 16 + (r & 15);  // in units of 8 floats
    int lo = 0, hi = N - 1;  // last document starting at or before row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (kvs[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const bool inside = row >= kvs[lo] && row < (int64_t)kvs[lo] + (cu[lo + 1] - cu[lo]);
    if (inside) {
      dk[i] = cast8(dk_acc + 2 * src);
      dv[i] = cast8(dv_acc + 2 * src);
    } else {
      dk[i] = make_uint4(0, 0, 0, 0);
      dv[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// main kernel arguments (the kernel itself is in msa_bwd_ws.cuh)
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
  int W;              // rows of the K/V axis (the dK, dV accumulators are [Hkv][W][128])
  int32_t* unit_ctr;  // next walk unit to hand out; 0 at launch
  float scale_log2;
  float scale;
  int32_t* status;
};

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
  if (stages & ~(uint32_t)(MSA_STAGE_ALL | MSA_BWD_DQ_FP32 | MSA_BWD_SELFTEST_HOLD_REDUCE))
    return MSA_ERR_INVALID_ARGUMENT;
  const bool dq_fp32 = (stages & MSA_BWD_DQ_FP32) != 0;
  const bool hold = (stages & MSA_BWD_SELFTEST_HOLD_REDUCE) != 0;
  if (hold && dq_fp32) return MSA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < bwd_ws_bytes(p, dq_fp32)) return MSA_ERR_INVALID_ARGUMENT;
  if ((rc = check_device_current())) return rc;
  int32_t sms = 0;
  if ((rc = sm_count_current(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t T = p->total_tokens, Hq = p->num_q_heads, W = p->kv_rows, Hkv = p->num_kv_heads;

  uint8_t* w = static_cast<uint8_t*>(ws);
  float* delta = reinterpret_cast<float*>(w);
  w += round_up(sizeof(float) * T * Hq, 256);
  float* dk_acc = reinterpret_cast<float*>(w);
  w += round_up(sizeof(float) * W * Hkv * kHeadDim, 256);
  float* dv_acc = reinterpret_cast<float*>(w);
  w += round_up(sizeof(float) * W * Hkv * kHeadDim, 256);
  const int64_t zero_n4 = (reinterpret_cast<float*>(w) - dk_acc) / 4;
  int32_t* unit_ctr = reinterpret_cast<int32_t*>(w);
  w += 256;
  float* dq_acc = dq_fp32 ? reinterpret_cast<float*>(w) : nullptr;

  // loads: Q/dO boxes of 8 tokens x 16 heads x 64 dims, K/V boxes of 64 keys x 64 dims;
  // reduce-adds: dQ boxes of 2 tokens x 16 heads x 64 dims (bf16, into the output)
  // or x 32 dims (fp32, into the accumulator), dK/dV of 32 keys x 32 dims (fp32)
  CUtensorMap tmQ, tmdO, tmK, tmV, tmdQ, tmdK, tmdV;
  bool ok = make_tmap_3d(&tmQ, q, false, T, Hq, 64, 16, 8) && make_tmap_3d(&tmdO, dout, false, T, Hq, 64, 16, 8) &&
            make_tmap_3d(&tmK, k, false, W, Hkv, 64, 1, 64) && make_tmap_3d(&tmV, v, false, W, Hkv, 64, 1, 64) &&
            (dq_fp32 ? make_tmap_3d(&tmdQ, dq_acc, true, T, Hq, 32, 16, 2)
                     : make_tmap_3d(&tmdQ, dq, false, T, Hq, 64, 16, 2)) &&
            make_tmap_3d(&tmdK, dk_acc, true, W * Hkv, 1, 32, 1, 32) &&
            make_tmap_3d(&tmdV, dv_acc, true, W * Hkv, 1, 32, 1, 32);
  if (!ok) return MSA_ERR_CUDA;

  const int64_t dq_n16 = T * Hq * kHeadDim * 2 / 16;  // 16-byte units of the bf16 dQ
  if (stages & MSA_STAGE_PREPROCESS)
    preprocess_kernel<<<sms * 8, 256, 0, st>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout), delta, T, (int)Hq,
        reinterpret_cast<float4*>(dk_acc), zero_n4,
        dq_fp32 ? reinterpret_cast<uint4*>(dq_acc) : reinterpret_cast<uint4*>(dq), dq_fp32 ? 2 * dq_n16 : dq_n16,
        d_status);
  if (stages & MSA_STAGE_MAIN) {
  auto* kernel = hold ? bwd_main_ws<false, true> : dq_fp32 ? bwd_main_ws<true> : bwd_main_ws<false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ws::SMEM) != cudaSuccess)
    return MSA_ERR_CUDA;
  const int64_t bound = msa_grid_launch_bound(task_cap, sms);
  const int grid = (int)(bound < sms ? (bound < 1 ? 1 : bound) : sms);
  MainArgs a;
  a.lse = lse; a.delta = delta; a.meta = task_meta; a.q_rows = task_q_rows; a.q_pos = task_q_pos; a.walk = walk;
  a.kv_doc_starts = p->kv_doc_starts; a.Hq = (int)Hq; a.W = (int)W; a.unit_ctr = unit_ctr; a.scale_log2 = p->softmax_scale * kLog2e;
  a.scale = p->softmax_scale; a.status = d_status;
  if ((rc = cuda_status(cudaMemsetAsync(unit_ctr, 0, sizeof(int32_t), st)))) return rc;
  kernel<<<grid, ws::kThreads, ws::SMEM, st>>>(tmQ, tmdO, tmK, tmV, tmdQ, tmdK, tmdV, a);
  }
  if (stages & MSA_STAGE_POSTPROCESS)
    postprocess_kernel<<<sms * 8, 256, 0, st>>>(
      reinterpret_cast<const float4*>(dk_acc), reinterpret_cast<const float4*>(dv_acc), reinterpret_cast<uint4*>(dk),
      reinterpret_cast<uint4*>(dv), W * Hkv * kHeadDim / 8, W, (int)Hkv, p->cu_seqlens,
      p->kv_doc_starts, p->num_docs, reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint4*>(dq), dq_n16,
      d_status);
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
