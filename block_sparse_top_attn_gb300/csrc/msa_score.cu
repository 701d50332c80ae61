// Block scorer and top-k selection: produces sel[Hi][NC][K] on the device from
// per-token index projections ("msa_bindings" page, MSAKernels.fmha_sm100, the
// scorer launcher; "msa_schedule" page, INDEX_DIM = 128 per index head).
//
// The pages name the scorer and its index dimension, not its score.  What is
// computed here (the reading this library documents):
//   pooled index query of each query chunk, pooled index key of each key
//   block: the mean of its tokens' index vectors within the document, an fp32
//   sum in token order divided by the token count (IEEE division), rounded to
//   bf16;
//   score(chunk, block) = fp32 dot product of the two pooled vectors summed in
//   ascending index-dim order (a product of two bf16 values is exact in fp32,
//   so a fused multiply-add rounds exactly as a multiply then an add would);
//   the chunk's diagonal block (the one holding its first query) comes first,
//   then the K-1 causal blocks before it with the highest scores, a tie going
//   to the lower block, then -1.
//
// Kernels: pool_kernel (one warp per chunk or block and index head; HBM-bound)
// and topk_kernel (a CTA scores 64 chunks against 64-block tiles with an 8 x 2
// register tile per thread, four dims per step, then each warp merges its
// rows' candidates into per-row top-(K-1) lists held one entry per lane).
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa_common.cuh"
#include "msa_host.cuh"

namespace msa {
namespace score {

constexpr int kDim = 128;        // index dim
constexpr int kRows = 64;        // chunks per CTA
constexpr int kCols = 64;        // blocks per tile
constexpr int kThreads = 256;
constexpr int kWarpRows = kRows / (kThreads / 32);  // rows (chunks) of one warp's register tile
// dynamic shared memory: pooled queries [kRows][kDim] and a transposed key
// tile [kDim][kCols] in fp32, then the rows' candidate ranges
constexpr uint32_t SMEM = (kRows * kDim + kDim * kCols) * 4 + 2 * kRows * 4;

// Largest d in [0, n) with off[d] <= x (off ascending, off[0] = 0 <= x).
__device__ __forceinline__ int doc_of(const int32_t* off, int n, int64_t x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct PoolArgs {
  const uint16_t* x;       // [T, Hi, 128] bf16
  uint16_t* out;           // [Hi, G, 128] bf16
  const int32_t* cu;
  const int32_t* goff;     // group offset of each document: chunk_off or blk_off, [N+1]
  int N, Hi, G, size;
  const int32_t* status;
};

// One warp per (group, index head); lane l owns dims 4l .. 4l+3.
__global__ void __launch_bounds__(256) pool_kernel(PoolArgs a) {
  if (status_bad(a.status)) return;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < (int64_t)a.G * a.Hi; w += nwarps) {
    const int g = (int)(w / a.Hi), hi = (int)(w % a.Hi);
    const int d = doc_of(a.goff, a.N + 1, g);
    const int len = a.cu[d + 1] - a.cu[d];
    const int first = (g - a.goff[d]) * a.size;
    const int n = min(a.size, len - first);
    const uint16_t* src = a.x + ((int64_t)(a.cu[d] + first) * a.Hi + hi) * kDim + lane * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int t = 0; t < n; ++t) {  // loads run ahead of the in-order sums
      const uint2 v = *reinterpret_cast<const uint2*>(src + (int64_t)t * a.Hi * kDim);
      acc[0] = __fadd_rn(acc[0], __uint_as_float(v.x << 16));
      acc[1] = __fadd_rn(acc[1], __uint_as_float(v.x & 0xFFFF0000u));
      acc[2] = __fadd_rn(acc[2], __uint_as_float(v.y << 16));
      acc[3] = __fadd_rn(acc[3], __uint_as_float(v.y & 0xFFFF0000u));
    }
    const float fn = (float)n;
    uint2 o;
    o.x = pack_bf16x2(__fdiv_rn(acc[0], fn), __fdiv_rn(acc[1], fn));
    o.y = pack_bf16x2(__fdiv_rn(acc[2], fn), __fdiv_rn(acc[3], fn));
    *reinterpret_cast<uint2*>(a.out + ((int64_t)hi * a.G + g) * kDim + lane * 4) = o;
  }
}

struct TopkArgs {
  const uint16_t* qpool;   // [Hi, NC, 128]
  const uint16_t* kpool;   // [Hi, NB, 128]
  const int32_t* chunk_off;
  const int32_t* blk_off;
  int32_t* sel;            // [Hi, NC, K]
  int N, Hi, NC, NB, K, B;
  int32_t* status;
};

// Candidate order: higher score first, then lower block.
__device__ __forceinline__ bool better(float sa, int ba, float sb, int bb) {
  return sa > sb || (sa == sb && ba < bb);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a) {
  extern __shared__ float smem_f[];
  float (*sq)[kDim] = reinterpret_cast<float (*)[kDim]>(smem_f);                 // pooled queries of the rows
  float (*sk)[kCols] = reinterpret_cast<float (*)[kCols]>(smem_f + kRows * kDim);  // a key tile, transposed
  int* s_lo = reinterpret_cast<int*>(smem_f + kRows * kDim + kDim * kCols);      // candidate blocks of each
  int* s_n = s_lo + kRows;                                                        // row: [lo, lo + n)
  if (status_bad(a.status)) return;
  const int hi = blockIdx.y, g0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rows: chunk, document, diagonal, candidate range [lo, lo + n)
  if (threadIdx.x < kRows) {
    const int g = g0 + threadIdx.x;
    int lo = 0, n = -1;
    if (g < a.NC) {
      const int d = doc_of(a.chunk_off, a.N + 1, g);
      const int diag = ((g - a.chunk_off[d]) * kChunk) / a.B;
      lo = a.blk_off[d];
      n = diag;
    }
    s_lo[threadIdx.x] = lo;
    s_n[threadIdx.x] = n;
  }
  for (int i = threadIdx.x; i < kRows * kDim / 2; i += kThreads) {
    const int r = i / (kDim / 2), c2 = i % (kDim / 2);
    uint32_t v = 0;
    if (g0 + r < a.NC) v = *reinterpret_cast<const uint32_t*>(a.qpool + ((int64_t)hi * a.NC + g0 + r) * kDim + c2 * 2);
    sq[r][2 * c2] = __uint_as_float(v << 16);
    sq[r][2 * c2 + 1] = __uint_as_float(v & 0xFFFF0000u);
  }
  __syncthreads();
  // the union of the rows' candidate ranges
  int blo = INT32_MAX, bhi = 0;
  for (int r = 0; r < kRows; ++r)
    if (s_n[r] > 0) {
      blo = min(blo, s_lo[r]);
      bhi = max(bhi, s_lo[r] + s_n[r]);
    }
  // per-row top-(K-1) lists: lane i holds entry i of each of the warp's rows
  const int keep = a.K - 1;
  float ls[kWarpRows];
  int lb[kWarpRows];
#pragma unroll
  for (int i = 0; i < kWarpRows; ++i) { ls[i] = -CUDART_INF_F; lb[i] = INT32_MAX; }
  for (int b0 = blo; b0 < bhi; b0 += kCols) {
    __syncthreads();  // the previous tile is no longer read
    {
      // thread t: block b0 + (t & 63), dims 32 * (t >> 6) .. + 31
      const int bb = threadIdx.x & 63, d0 = (threadIdx.x >> 6) * 32;
      const int r = b0 + bb;
      const uint4* src = reinterpret_cast<const uint4*>(a.kpool + ((int64_t)hi * a.NB + min(r, a.NB - 1)) * kDim + d0);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 v = r < a.NB ? src[q4] : make_uint4(0, 0, 0, 0);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sk[d0 + q4 * 8 + 2 * e][bb] = __uint_as_float(w[e] << 16);
          sk[d0 + q4 * 8 + 2 * e + 1][bb] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
      }
    }
    __syncthreads();
    // kWarpRows rows (from kWarpRows * warp) x 2 blocks (b0 + 2 lane, + 1),
    // summed over the dims in ascending order (four dims per step: a row's
    // four query values in one 16-byte load that every lane shares, so twelve
    // shared-memory loads feed 64 FMAs)
    float s[kWarpRows][2];
#pragma unroll
    for (int i = 0; i < kWarpRows; ++i) s[i][0] = s[i][1] = 0.f;
#pragma unroll 2
    for (int d = 0; d < kDim; d += 4) {
      float2 kv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) kv[e] = *reinterpret_cast<const float2*>(&sk[d + e][2 * lane]);
#pragma unroll
      for (int i = 0; i < kWarpRows; ++i) {
        const float4 q4 = *reinterpret_cast<const float4*>(&sq[kWarpRows * warp + i][d]);
        const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s[i][0] = __fmaf_rn(qv[e], kv[e].x, s[i][0]);
          s[i][1] = __fmaf_rn(qv[e], kv[e].y, s[i][1]);
        }
      }
    }
    // merge each row's candidates of this tile into its list
#pragma unroll
    for (int i = 0; i < kWarpRows; ++i) {
      const int r = kWarpRows * warp + i;
      const int lo = s_lo[r], n = s_n[r];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int bidx = b0 + 2 * lane + jj;
        const float sc = s[i][jj];
        bool cand = keep > 0 && bidx >= lo && bidx < lo + n;
        // threshold: the current last kept entry
        float ts = __shfl_sync(0xffffffffu, ls[i], max(keep - 1, 0));
        int tb = __shfl_sync(0xffffffffu, lb[i], max(keep - 1, 0));
        unsigned m = __ballot_sync(0xffffffffu, cand && better(sc, bidx, ts, tb));
        while (m) {
          const int src = __ffs(m) - 1;
          m &= m - 1;
          const float xs = __shfl_sync(0xffffffffu, sc, src);
          const int xb = __shfl_sync(0xffffffffu, bidx, src);
          ts = __shfl_sync(0xffffffffu, ls[i], keep - 1);
          tb = __shfl_sync(0xffffffffu, lb[i], keep - 1);
          if (!better(xs, xb, ts, tb)) continue;  // the threshold rose past it
          // position = number of kept entries better than the candidate
          const unsigned ahead = __ballot_sync(0xffffffffu, lane < keep && better(ls[i], lb[i], xs, xb));
          const int pos = __popc(ahead);
          const float us = __shfl_up_sync(0xffffffffu, ls[i], 1);
          const int ub = __shfl_up_sync(0xffffffffu, lb[i], 1);
          if (lane < keep) {
            if (lane == pos) { ls[i] = xs; lb[i] = xb; }
            else if (lane > pos) { ls[i] = us; lb[i] = ub; }
          }
        }
      }
    }
  }
  // write the rows: diagonal, the kept blocks (document-local), -1 pads
#pragma unroll
  for (int i = 0; i < kWarpRows; ++i) {
    const int r = kWarpRows * warp + i, g = g0 + r;
    if (g >= a.NC) continue;
    const int lo = s_lo[r];
    int32_t* row = a.sel + ((int64_t)hi * a.NC + g) * a.K;
    if (lane == 0) row[0] = s_n[r];
    if (lane < keep) row[1 + lane] = lb[i] == INT32_MAX ? -1 : lb[i] - lo;
  }
}

}  // namespace score
}  // namespace msa

using namespace msa;

extern "C" int msa_select_topk(const msa_problem* p, const uint16_t* q_index, const uint16_t* k_index, int32_t* sel,
                               int32_t* d_status, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (!q_index || !k_index || !sel || !d_status || !ws) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_index) || !aligned16(k_index) || !aligned16(sel) || !aligned16(d_status) || !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < select_ws_bytes(p)) return MSA_ERR_INVALID_ARGUMENT;
  if ((rc = check_device_current())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = p->num_docs, NB = p->num_blocks, NC = p->num_chunks, Hi = p->num_index_heads;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* blk_off = reinterpret_cast<int32_t*>(w);
  int32_t* chunk_off = blk_off + (N + 1);
  w += round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  uint16_t* qpool = reinterpret_cast<uint16_t*>(w);
  w += round_up(sizeof(uint16_t) * Hi * NC * score::kDim, 256);
  uint16_t* kpool = reinterpret_cast<uint16_t*>(w);
  if ((rc = launch_layout(p, blk_off, chunk_off, d_status, st))) return rc;
  int32_t sms = 0;
  if ((rc = sm_count_current(&sms))) return rc;
  score::PoolArgs pa{q_index, qpool, p->cu_seqlens, chunk_off, N, Hi, NC, kChunk, d_status};
  score::pool_kernel<<<sms * 8, 256, 0, st>>>(pa);
  score::PoolArgs pk{k_index, kpool, p->cu_seqlens, blk_off, N, Hi, NB, p->block_size, d_status};
  score::pool_kernel<<<sms * 8, 256, 0, st>>>(pk);
  score::TopkArgs ta{qpool, kpool, chunk_off, blk_off, sel, N, Hi, NC, NB, p->topk, p->block_size, d_status};
  if ((rc = cuda_status(cudaFuncSetAttribute(score::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)score::SMEM))))
    return rc;
  score::topk_kernel<<<dim3((unsigned)((NC + score::kRows - 1) / score::kRows), Hi), score::kThreads, score::SMEM,
                       st>>>(ta);
  return cuda_status(cudaGetLastError());
}
