// MSA block-sparse attention forward on sm_103a ("msa_bindings" page,
// sparse_atten_func, the flat forward): per (index head, query chunk) the 128
// rows (8 tokens x 16 q-heads) attend the chunk's selected key blocks
// causally.  Two passes over the selected blocks with tcgen05 GEMMs:
//   pass 1  S = Q K^T                 -> running max and sum of exp2 (log2 LSE)
//   pass 2  S = Q K^T, P = exp2(S - LSE), O += P V   (P as bf16 in smem)
// O is written as bf16 and LSE in natural log, the form the backward consumes.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa_common.cuh"
#include "msa_host.cuh"
#include "msa_tmap.cuh"

namespace msa {

namespace fwd {
constexpr uint32_t OFF_Q = 0;       // [2 halves][128 rows][128 B]
constexpr uint32_t OFF_K = 32768;   // [2 halves][64 keys][128 B]
constexpr uint32_t OFF_V = 49152;
constexpr uint32_t OFF_P = 65536;   // [128 rows][64 keys bf16]
constexpr uint32_t OFF_BAR = 81920;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_S = 0, COL_O = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace fwd

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct FwdArgs {
  const int32_t* sel;
  const int32_t* cu;
  const int32_t* chunk_off;
  uint16_t* o;
  float* lse;
  int N, NC, K, Hi, Hq;
  float scale_log2;
  int32_t* status;
};

__device__ __forceinline__ int doc_of_chunk(const int32_t* chunk_off, int n, int g) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (chunk_off[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(128, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const int32_t* kv_doc_starts, FwdArgs a) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_load + 2);
  int* s_blocks = reinterpret_cast<int*>(bar_load + 4);  // up to 32 selected blocks
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
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
  constexpr uint32_t ID_O = idesc_bf16_f32(128, 128, false, true);
  uint32_t ph_load = 0, ph_mma = 0;
  bool aborted = status_bad(a.status);
  const int64_t items = (int64_t)a.Hi * a.NC;
  for (int64_t w = blockIdx.x; w < items && !aborted; w += gridDim.x) {
    const int hi = (int)(w / a.NC), g = (int)(w % a.NC);
    const int d = doc_of_chunk(a.chunk_off, a.N + 1, g);
    const int c = g - a.chunk_off[d];
    const int len = a.cu[d + 1] - a.cu[d];
    const int tok0 = a.cu[d] + c * 8;
    const int qcount = min(8, len - c * 8);
    const int slot = tid >> 4, hh = tid & 15;
    const int qpos = slot < qcount ? c * 8 + slot : -1;
    if (tid == 0) {
      int nb = 0;
      for (int j = 0; j < a.K; ++j) {
        const int b = a.sel[((int64_t)hi * a.NC + g) * a.K + j];
        if (b >= 0) s_blocks[nb++] = b;
      }
      s_blocks[32] = nb;
    }
    __syncthreads();
    const int nblk = s_blocks[32];
    const int kv0 = kv_doc_starts[d];
    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool q_loaded = false;
    for (int pass = 0; pass < 2 && !aborted; ++pass) {
      float lse2 = m_run + lg2_approx(l_run);
      for (int j = 0; j < nblk; ++j) {
        const int b = s_blocks[j];
        const int kvrow = kv0 + b * 64;
        if (tid == 0) {
          const uint32_t bytes = (q_loaded ? 0u : 32768u) + 16384u + (pass == 1 ? 16384u : 0u);
          mbar_arrive_expect_tx(bar_load, bytes);
          if (!q_loaded) {
            tma_load_3d(sm + OFF_Q, &tmQ, bar_load, 0, hi * 16, tok0);
            tma_load_3d(sm + OFF_Q + 16384, &tmQ, bar_load, 64, hi * 16, tok0);
          }
          tma_load_3d(sm + OFF_K, &tmK, bar_load, 0, hi, kvrow);
          tma_load_3d(sm + OFF_K + 8192, &tmK, bar_load, 64, hi, kvrow);
          if (pass == 1) {
            tma_load_3d(sm + OFF_V, &tmV, bar_load, 0, hi, kvrow);
            tma_load_3d(sm + OFF_V + 8192, &tmV, bar_load, 64, hi, kvrow);
          }
        }
        q_loaded = true;
        if (!mbar_wait(bar_load, ph_load, a.status)) aborted = true;
        ph_load ^= 1;
        if (__syncthreads_or(aborted)) { aborted = true; break; }
        if (tid == 0) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
            umma_bf16(tmem + COL_S, sdesc_sw128(sbase + OFF_Q + half * 16384 + sub, 16, 1024),
                      sdesc_sw128(sbase + OFF_K + half * 8192 + sub, 16, 1024), ID_S, kk > 0);
          }
          umma_commit(bar_mma);
        }
        if (!mbar_wait(bar_mma, ph_mma, a.status)) aborted = true;
        ph_mma ^= 1;
        if (__syncthreads_or(aborted)) { aborted = true; break; }
        tc_fence_after();
        uint32_t pk[32];
        float bmax = -CUDART_INF_F;
        float xs[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t sv[16];
          tmem_ld16(tmem + lane_base + COL_S + c0, sv);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const bool valid = qpos >= 0 && b * 64 + c0 + e <= qpos;
            const float x = valid ? __uint_as_float(sv[e]) * a.scale_log2 : -CUDART_INF_F;
            xs[c0 + e] = x;
            bmax = fmaxf(bmax, x);
          }
        }
        if (pass == 0) {
          const float m_new = fmaxf(m_run, bmax);
          if (m_new > -CUDART_INF_F) {
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < 64; ++e) s += ex2_approx(xs[e] - m_new);
            l_run = l_run * ex2_approx(m_run - m_new) + s;
            m_run = m_new;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; e += 2)
            pk[e >> 1] = pack_bf16x2(xs[e] > -CUDART_INF_F ? ex2_approx(xs[e] - lse2) : 0.f,
                                     xs[e + 1] > -CUDART_INF_F ? ex2_approx(xs[e + 1] - lse2) : 0.f);
          uint8_t* prow = sm + OFF_P + tid * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4*>(prow + ((cc ^ (tid & 7)) << 4)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          fence_async_smem();
          tc_fence_before();
          __syncthreads();
          if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + COL_O, sdesc_sw128(sbase + OFF_P + kk * 32, 16, 1024),
                        sdesc_sw128(sbase + OFF_V + kk * 2048, 8192, 1024), ID_O, (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit(bar_mma);
          }
          if (!mbar_wait(bar_mma, ph_mma, a.status)) aborted = true;
          ph_mma ^= 1;
          if (__syncthreads_or(aborted)) { aborted = true; break; }
          tc_fence_after();
        }
      }
    }
    if (aborted) break;
    // epilogue: O row -> bf16 global, LSE natural log.  TMEM loads are
    // warp-collective, so every thread loads and only real rows store.
    {
      const int64_t row = (int64_t)(tok0 + slot) * a.Hq + hi * 16 + hh;
      if (qpos >= 0) a.lse[row] = l_run > 0.f ? (m_run + lg2_approx(l_run)) * kLn2 : -CUDART_INF_F;
      uint4* dst = reinterpret_cast<uint4*>(a.o + row * 128);
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t v[16];
        if (nblk > 0) {
          tmem_ld16(tmem + lane_base + COL_O + c0, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0u;
        }
        if (qpos >= 0) {
          dst[c0 / 8] = make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                                   pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                                   pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                                   pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
          dst[c0 / 8 + 1] = make_uint4(pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9])),
                                       pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11])),
                                       pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13])),
                                       pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15])));
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// defined in msa_tables.cu
__global__ void layout_kernel(const int32_t* cu, const int32_t* kvs, int N, int T, int W, int NB, int NC,
                              int32_t* blk_off, int32_t* chunk_off, int32_t* status);

}  // namespace msa

using namespace msa;

extern "C" int msa_fwd(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* sel, uint16_t* o, float* lse, int32_t* d_status, void* ws, size_t ws_bytes,
                       void* stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  const void* ptrs[] = {q, k, v, sel, o, lse, d_status, ws};
  for (const void* x : ptrs)
    if (!x || !aligned16(x)) return MSA_ERR_INVALID_ARGUMENT;
  const int N = p->num_docs;
  if (ws_bytes < round_up(sizeof(int32_t) * 2 * (N + 1), 256)) return MSA_ERR_INVALID_ARGUMENT;
  if ((rc = check_device_current())) return rc;
  int32_t sms = 0;
  if ((rc = sm_count_current(&sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t T = p->total_tokens, Hq = p->num_q_heads, W = p->kv_rows, Hkv = p->num_kv_heads;
  int32_t* blk_off = static_cast<int32_t*>(ws);
  int32_t* chunk_off = blk_off + (N + 1);
  CUtensorMap tmQ, tmK, tmV;
  if (!(make_tmap_3d(&tmQ, q, false, T, Hq, 64, 16, 8) && make_tmap_3d(&tmK, k, false, W, Hkv, 64, 1, 64) &&
        make_tmap_3d(&tmV, v, false, W, Hkv, 64, 1, 64)))
    return MSA_ERR_CUDA;
  layout_kernel<<<1, 1024, 0, st>>>(p->cu_seqlens, p->kv_doc_starts, N, p->total_tokens, p->kv_rows,
                                    p->num_blocks, p->num_chunks, blk_off, chunk_off, d_status);
  if (cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fwd::SMEM) != cudaSuccess)
    return MSA_ERR_CUDA;
  FwdArgs a;
  a.sel = sel; a.cu = p->cu_seqlens; a.chunk_off = chunk_off; a.o = o; a.lse = lse; a.N = N;
  a.NC = p->num_chunks; a.K = p->topk; a.Hi = p->num_index_heads; a.Hq = (int)Hq;
  a.scale_log2 = p->softmax_scale * fwd::kLog2e; a.status = d_status;
  const int64_t items = (int64_t)p->num_index_heads * p->num_chunks;
  // ~82 KB of shared memory: two CTAs per SM
  const int grid = (int)(items < 2 * sms ? items : 2 * sms);
  fwd_kernel<<<grid, 128, fwd::SMEM, st>>>(tmQ, tmK, tmV, p->kv_doc_starts, a);
  return cuda_status(cudaGetLastError());
}
