// Index tables of the MSA backward: the key-block -> query CSR (msa_build_k2q),
// the task rows and CTA walk (msa_build_tasks), and the host-side helpers of
// the C ABI (validation, memoised device queries, workspace sizing, walk rule).
//
// Both builds are deterministic: counts are order-independent sums, and every
// position-dependent write is ordered by a sequential walk over query chunks
// within a scatter group plus exclusive prefix sums across groups.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "msa_common.cuh"
#include "msa_host.cuh"

namespace msa {

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
int check_problem(const msa_problem* p) {
  if (!p || !p->cu_seqlens || !p->kv_doc_starts) return MSA_ERR_INVALID_ARGUMENT;
  if (p->num_docs < 1 || p->total_tokens < 1 || p->kv_rows < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(p->cu_seqlens) || !aligned16(p->kv_doc_starts)) return MSA_ERR_INVALID_ARGUMENT;
  if (p->num_index_heads < 1 || p->num_kv_heads < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (p->head_dim != kHeadDim || p->block_size != kBlock || p->query_chunk != kChunk)
    return MSA_ERR_UNSUPPORTED_SHAPE;
  if (p->num_kv_heads != p->num_index_heads || p->num_q_heads != kGroup * p->num_index_heads)
    return MSA_ERR_UNSUPPORTED_SHAPE;
  if (p->topk < 1 || p->topk > kMaxTopk) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (p->num_blocks < 1 || p->num_chunks < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (p->num_blocks > kMaxRows) return MSA_ERR_UNSUPPORTED_SHAPE;
  // counts implied by T alone bound the per-document sums
  const int64_t T = p->total_tokens, N = p->num_docs;
  if (p->num_chunks < (T + kChunk - 1) / kChunk || p->num_chunks > T / kChunk + N) return MSA_ERR_INVALID_ARGUMENT;
  if (p->num_blocks < (T + kBlock - 1) / kBlock || p->num_blocks > T / kBlock + N) return MSA_ERR_INVALID_ARGUMENT;
  if (!(p->softmax_scale > 0.f)) return MSA_ERR_INVALID_ARGUMENT;
  return MSA_OK;
}

size_t k2q_ws_bytes(const msa_problem* p) {
  const int64_t Hi = p->num_index_heads, NB = p->num_blocks, NC = p->num_chunks, N = p->num_docs;
  const int64_t nS = (NC + k2q_group_chunks(NC) - 1) / k2q_group_chunks(NC);
  size_t b = round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  b += round_up(sizeof(int32_t) * Hi * nS * NB, 256);
  b += round_up(sizeof(int32_t) * Hi * NB, 256);
  return b;
}

size_t select_ws_bytes(const msa_problem* p) {
  const int64_t Hi = p->num_index_heads, NB = p->num_blocks, NC = p->num_chunks, N = p->num_docs;
  size_t b = round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  b += round_up(sizeof(uint16_t) * Hi * NC * kHeadDim, 256);   // pooled index queries
  b += round_up(sizeof(uint16_t) * Hi * NB * kHeadDim, 256);   // pooled index keys
  return b;
}

static constexpr int kScanSeg = 2048;  // elements per block of the multi-block scan

size_t tasks_ws_bytes(const msa_problem* p, int32_t tile_chunks) {
  const int64_t Hi = p->num_index_heads, NB = p->num_blocks, NC = p->num_chunks, N = p->num_docs;
  const int64_t n = Hi * num_tiles(NC, tile_chunks) * NB;
  size_t b = round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  b += round_up(sizeof(int32_t) * n, 256) * 2;
  b += round_up(sizeof(int32_t) * ((n + kScanSeg - 1) / kScanSeg + 1), 256);
  return b;
}

size_t bwd_ws_bytes(const msa_problem* p) {
  const int64_t T = p->total_tokens, Hq = p->num_q_heads, W = p->kv_rows, Hkv = p->num_kv_heads;
  size_t b = round_up(sizeof(float) * T * Hq, 256);                 // D
  b += 2 * round_up(sizeof(float) * W * Hkv * kHeadDim, 256);       // dK, dV accumulators
  b += 256;                                                          // walk-unit counter
  return b;
}

namespace {
struct DevInfo {
  bool valid = false;
  int major = 0, minor = 0, sms = 0;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int dev_info(int32_t device, DevInfo* out) {
  if (device < 0 || device >= kMaxDevices) return MSA_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[device];
  if (!d.valid) {
    if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      cudaGetLastError();
      return MSA_ERR_CUDA;
    }
    d.valid = true;
  }
  *out = d;
  return MSA_OK;
}
}  // namespace

int sm_count_current(int32_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  DevInfo d;
  int rc = dev_info(dev, &d);
  if (rc) return rc;
  *out = d.sms;
  return MSA_OK;
}

int check_device_current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  DevInfo d;
  int rc = dev_info(dev, &d);
  if (rc) return rc;
  return (d.major == 10 && d.minor == 3) ? MSA_OK : MSA_ERR_UNSUPPORTED_DEVICE;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
// Largest d in [0, n) with off[d] <= x (off ascending, off[0] = 0 <= x).
__device__ __forceinline__ int upper_index(const int32_t* off, int n, int64_t x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = warp_sums[lane];
    int t = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_sums[lane] = t - s;
    if (lane == 31) *total = t;
  }
  __syncthreads();
  int r = x - v + warp_sums[w];
  __syncthreads();
  return r;
}

// Document layout: blk_off[d], chunk_off[d] for d in [0, N] and consistency checks.
__global__ void __launch_bounds__(1024) layout_kernel(const int32_t* cu, const int32_t* kvs, int N, int T, int W,
                                                       int NB, int NC, int32_t* blk_off, int32_t* chunk_off,
                                                       int32_t* status) {
  __shared__ int ws[32];
  __shared__ int tot;
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  int carry_b = 0, carry_c = 0;
  for (int base = 0; base < N; base += 1024) {
    const int d = base + threadIdx.x;
    int nb = 0, nc = 0;
    if (d < N) {
      const int a = cu[d], b = cu[d + 1];
      const int len = b - a;
      if (len <= 0 || (d == 0 && a != 0) || (d == N - 1 && b != T)) bad = 1;
      const int k0 = kvs[d];
      if (k0 < 0 || (int64_t)k0 + len > W) bad = 1;
      if (d + 1 < N && (int64_t)k0 + len > kvs[d + 1]) bad = 1;
      nb = len > 0 ? (len + kBlock - 1) / kBlock : 0;
      nc = len > 0 ? (len + kChunk - 1) / kChunk : 0;
    }
    const int eb = block_excl_scan(nb, ws, &tot);
    const int tb = tot;
    const int ec = block_excl_scan(nc, ws, &tot);
    const int tc = tot;
    if (d < N) {
      blk_off[d] = carry_b + eb;
      chunk_off[d] = carry_c + ec;
    }
    carry_b += tb;
    carry_c += tc;
  }
  if (threadIdx.x == 0) {
    blk_off[N] = carry_b;
    chunk_off[N] = carry_c;
    if (carry_b != NB || carry_c != NC) bad = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0 && bad) set_status(status, MSA_ERR_INVALID_DOCUMENTS);
}

// ---------------------------------------------------------------------------
// k2q CSR build
// ---------------------------------------------------------------------------
struct K2QArgs {
  const int32_t* sel;
  const int32_t* cu;
  const int32_t* blk_off;
  const int32_t* chunk_off;
  int32_t* cnt;       // [Hi][nS][NB] group counts, then exclusive group offsets
  int32_t* totals;    // [Hi][NB]
  int32_t* row_ptr;   // [Hi][NB+1]
  int32_t* q_indices; // [Hi][edge_cap]
  int64_t edge_cap;
  int N, NB, NC, K, SG, nS;
  int32_t* status;
};

// Rows [r_lo, r_hi) of the documents that group s's chunks belong to.
__device__ __forceinline__ void group_rows(const K2QArgs& a, int s, int* d_first, int* r_lo, int* r_hi) {
  const int g0 = s * a.SG;
  const int g1 = min(a.NC, g0 + a.SG) - 1;
  const int d0 = upper_index(a.chunk_off, a.N + 1, g0);
  const int d1 = upper_index(a.chunk_off, a.N + 1, g1);
  *d_first = d0;
  *r_lo = a.blk_off[d0];
  *r_hi = a.blk_off[d1 + 1];
}

// Per (scatter group, index head): validate the selection and count query
// entries per key-block row.  One warp per chunk, one lane per slot.
__global__ void __launch_bounds__(256) k2q_count_kernel(K2QArgs a) {
  extern __shared__ int hist[];
  if (status_bad(a.status)) return;
  const int s = blockIdx.x, hi = blockIdx.y;
  int d_first, r_lo, r_hi;
  group_rows(a, s, &d_first, &r_lo, &r_hi);
  for (int i = threadIdx.x; i < r_hi - r_lo; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g_end = min(a.NC, (s + 1) * a.SG);
  for (int g = s * a.SG + w; g < g_end; g += blockDim.x >> 5) {
    const int d = upper_index(a.chunk_off, a.N + 1, g);
    const int c = g - a.chunk_off[d];
    const int len_d = a.cu[d + 1] - a.cu[d];
    const int nb_d = a.blk_off[d + 1] - a.blk_off[d];
    const int len = min(kChunk, len_d - c * kChunk);
    int b = -1;
    if (lane < a.K) b = a.sel[((int64_t)hi * a.NC + g) * a.K + lane];
    bool bad = false;
    if (b != -1 && (b < 0 || b >= nb_d || (int64_t)b * kBlock > (int64_t)c * kChunk)) bad = true;
    const int key = (b >= 0 && !bad) ? b : -2 - lane;
    const unsigned same = __match_any_sync(0xffffffffu, key);
    if (__popc(same) > 1) bad = true;
    if (bad) set_status(a.status, MSA_ERR_INVALID_SELECTION);
    if (b >= 0 && !bad) atomicAdd(&hist[a.blk_off[d] + b - r_lo], len);
  }
  __syncthreads();
  int32_t* out = a.cnt + ((int64_t)hi * a.nS + s) * a.NB;
  for (int r = threadIdx.x; r < a.NB; r += blockDim.x)
    out[r] = (r >= r_lo && r < r_hi) ? hist[r - r_lo] : 0;
}

// Per (index head, row): exclusive offsets of each group within the row, and
// the row total.
__global__ void k2q_group_offsets_kernel(K2QArgs a, int Hi) {
  if (status_bad(a.status)) return;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)Hi * a.NB) return;
  const int hi = (int)(i / a.NB), r = (int)(i % a.NB);
  int run = 0;
  for (int s = 0; s < a.nS; ++s) {
    int32_t* c = a.cnt + ((int64_t)hi * a.nS + s) * a.NB + r;
    const int v = *c;
    *c = run;
    run += v;
  }
  a.totals[(int64_t)hi * a.NB + r] = run;
}

// Per index head: row_ptr = exclusive scan of the row totals.
__global__ void __launch_bounds__(1024) k2q_row_ptr_kernel(K2QArgs a) {
  __shared__ int ws[32];
  __shared__ int tot;
  if (status_bad(a.status)) return;
  const int hi = blockIdx.x;
  const int32_t* t = a.totals + (int64_t)hi * a.NB;
  int32_t* rp = a.row_ptr + (int64_t)hi * (a.NB + 1);
  int64_t carry = 0;
  for (int base = 0; base < a.NB; base += 1024) {
    const int r = base + threadIdx.x;
    const int v = r < a.NB ? t[r] : 0;
    const int e = block_excl_scan(v, ws, &tot);
    if (r < a.NB) rp[r] = (int32_t)(carry + e);
    carry += tot;
  }
  if (threadIdx.x == 0) {
    rp[a.NB] = (int32_t)carry;
    if (carry > a.edge_cap) set_status(a.status, MSA_ERR_CAPACITY);
  }
}

// Per (scatter group, index head), one warp: walk the group's chunks in order
// and append each chunk's positions to the rows it selected.
__global__ void __launch_bounds__(32) k2q_scatter_kernel(K2QArgs a) {
  extern __shared__ int cursor[];
  if (status_bad(a.status)) return;
  const int s = blockIdx.x, hi = blockIdx.y, lane = threadIdx.x;
  int d, r_lo, r_hi;
  group_rows(a, s, &d, &r_lo, &r_hi);
  const int32_t* rp = a.row_ptr + (int64_t)hi * (a.NB + 1);
  const int32_t* off = a.cnt + ((int64_t)hi * a.nS + s) * a.NB;
  for (int r = r_lo + lane; r < r_hi; r += 32) cursor[r - r_lo] = rp[r] + off[r];
  __syncwarp();
  int32_t* qi = a.q_indices + (int64_t)hi * a.edge_cap;
  const int g_begin = s * a.SG, g_end = min(a.NC, (s + 1) * a.SG);
  int next_b = -1;
  if (g_begin < g_end && lane < a.K) next_b = a.sel[((int64_t)hi * a.NC + g_begin) * a.K + lane];
  for (int g = g_begin; g < g_end; ++g) {
    const int b = next_b;
    if (g + 1 < g_end && lane < a.K) next_b = a.sel[((int64_t)hi * a.NC + g + 1) * a.K + lane];
    while (a.chunk_off[d + 1] <= g) ++d;
    const int c = g - a.chunk_off[d];
    const int len = min(kChunk, a.cu[d + 1] - a.cu[d] - c * kChunk);
    int p = -1;
    if (b >= 0) {
      const int row = a.blk_off[d] + b - r_lo;
      p = cursor[row];
      cursor[row] = p + len;
    }
    __syncwarp();
    if (p >= 0 && (int64_t)p + len <= a.edge_cap) {
      int32_t* dst = qi + p;
      const int v0 = c * kChunk;
      if (len == kChunk && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
        // a full chunk at a 16-byte boundary: two vector stores
        reinterpret_cast<int4*>(dst)[0] = make_int4(v0, v0 + 1, v0 + 2, v0 + 3);
        reinterpret_cast<int4*>(dst)[1] = make_int4(v0 + 4, v0 + 5, v0 + 6, v0 + 7);
      } else {
        for (int i = 0; i < len; ++i) dst[i] = v0 + i;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// task build
// ---------------------------------------------------------------------------
struct TaskArgs {
  const int32_t* row_ptr;
  const int32_t* q_indices;
  const int32_t* cu;
  const int32_t* blk_off;
  const int32_t* chunk_off;
  int32_t* tcnt;   // [Hi][ntiles][NB] task counts
  int32_t* toff;   // exclusive scan of tcnt
  int32_t* bsum;   // per scan block sums
  int32_t* meta;
  int32_t* q_rows;
  int32_t* q_pos;
  int32_t* walk;
  int64_t edge_cap, task_cap;
  int N, NB, NC, Hi, tile_chunks, ntiles, num_sms;
  int32_t* status;
};

__device__ __forceinline__ int task_tile(const TaskArgs& a, int64_t g) {
  return a.tile_chunks > 0 ? (int)(g / a.tile_chunks) : 0;
}

// A warp per (index head, row): count the row's groups per query tile.
__global__ void __launch_bounds__(256) task_count_kernel(TaskArgs a) {
  if (status_bad(a.status)) return;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)a.Hi * a.NB) return;
  const int hi = (int)(wid / a.NB), r = (int)(wid % a.NB);
  const int32_t* rp = a.row_ptr + (int64_t)hi * (a.NB + 1);
  const int lo = rp[r], end = rp[r + 1];
  if (lo < 0 || end < lo || end > a.edge_cap) {
    if (lane == 0) set_status(a.status, MSA_ERR_INVALID_ARGUMENT);
    return;
  }
  const int d = upper_index(a.blk_off, a.N + 1, r);
  const int len_d = a.cu[d + 1] - a.cu[d];
  const int ngroups = (end - lo + kChunk - 1) / kChunk;
  const int32_t* qi = a.q_indices + (int64_t)hi * a.edge_cap;
  for (int k = lane; k < ngroups; k += 32) {
    const int pos = qi[lo + k * kChunk];
    if (pos < 0 || pos >= len_d) {
      set_status(a.status, MSA_ERR_INVALID_ARGUMENT);
      continue;
    }
    const int t = task_tile(a, (int64_t)a.chunk_off[d] + pos / kChunk);
    atomicAdd(&a.tcnt[((int64_t)hi * a.ntiles + t) * a.NB + r], 1);
  }
}

// Multi-block exclusive scan, phase 1: per-segment sums.
__global__ void __launch_bounds__(1024) scan_reduce_kernel(const int32_t* in, int64_t n, int32_t* bsum,
                                                            const int32_t* status) {
  __shared__ int ws[32];
  __shared__ int tot;
  if (status_bad(status)) return;
  const int64_t base = (int64_t)blockIdx.x * kScanSeg;
  int v = 0;
  for (int i = threadIdx.x; i < kScanSeg; i += 1024)
    if (base + i < n) v += in[base + i];
  block_excl_scan(v, ws, &tot);
  if (threadIdx.x == 0) bsum[blockIdx.x] = tot;
}

// Phase 2: scan the segment sums (one block); the total is the task count,
// which sizes the CTA walk.
__global__ void __launch_bounds__(1024) scan_bsums_walk_kernel(int32_t* bsum, int nblk, TaskArgs a) {
  __shared__ int ws[32];
  __shared__ int tot;
  if (status_bad(a.status)) return;
  int64_t carry = 0;
  for (int base = 0; base < nblk; base += 1024) {
    const int i = base + threadIdx.x;
    const int v = i < nblk ? bsum[i] : 0;
    const int e = block_excl_scan(v, ws, &tot);
    if (i < nblk) bsum[i] = (int32_t)(carry + e);
    carry += tot;
  }
  if (threadIdx.x == 0) {
    const int64_t n = carry;
    if (n > a.task_cap) set_status(a.status, MSA_ERR_CAPACITY);
    const int R = n < 2400 ? 4 : 64;
    const int64_t full = n / R, tail = n - full * R;
    const int64_t grid = full + (tail < a.num_sms ? tail : a.num_sms);
    a.walk[MSA_WALK_ROWS] = (int32_t)n;
    a.walk[MSA_WALK_ROWS_PER_CTA] = R;
    a.walk[MSA_WALK_FULL] = (int32_t)full;
    a.walk[MSA_WALK_TAIL] = (int32_t)tail;
    a.walk[MSA_WALK_GRID] = (int32_t)grid;
    a.walk[MSA_WALK_SMS] = a.num_sms;
    a.walk[6] = 0;
    a.walk[7] = 0;
  }
}

// Phase 3: exclusive scan within each segment plus the segment offset.
__global__ void __launch_bounds__(1024) scan_apply_kernel(const int32_t* in, int64_t n, const int32_t* bsum,
                                                           int32_t* out, const int32_t* status) {
  __shared__ int ws[32];
  __shared__ int tot;
  if (status_bad(status)) return;
  const int64_t base = (int64_t)blockIdx.x * kScanSeg;
  int carry = bsum[blockIdx.x];
  for (int i0 = 0; i0 < kScanSeg; i0 += 1024) {
    const int64_t i = base + i0 + threadIdx.x;
    const int v = i < n ? in[i] : 0;
    const int e = block_excl_scan(v, ws, &tot);
    if (i < n) out[i] = carry + e;
    carry += tot;
  }
}

// A warp per (index head, row): emit the row's tasks.  Groups of one query
// tile are consecutive in the row, so a task's index is the tile's offset for
// this row plus its rank within the tile's run.
__global__ void __launch_bounds__(256) task_emit_kernel(TaskArgs a) {
  if (status_bad(a.status)) return;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)a.Hi * a.NB) return;
  const int hi = (int)(wid / a.NB), r = (int)(wid % a.NB);
  const int32_t* rp = a.row_ptr + (int64_t)hi * (a.NB + 1);
  const int lo = rp[r], end = rp[r + 1];
  const int d = upper_index(a.blk_off, a.N + 1, r);
  const int b = r - a.blk_off[d];
  const int tok0 = a.cu[d];
  const int ngroups = (end - lo + kChunk - 1) / kChunk;
  const int32_t* qi = a.q_indices + (int64_t)hi * a.edge_cap;
  int prev_tile = -1, prev_start = 0;  // carried across warp iterations
  for (int k0 = 0; k0 < ngroups; k0 += 32) {
    const int k = k0 + lane;
    const bool act = k < ngroups;
    int s = 0, cnt = 0, tile = -1, pos0 = 0;
    if (act) {
      s = lo + k * kChunk;
      cnt = min(kChunk, end - s);
      pos0 = qi[s];
      tile = task_tile(a, (int64_t)a.chunk_off[d] + pos0 / kChunk);
    }
    int left_tile = __shfl_up_sync(0xffffffffu, tile, 1);
    if (lane == 0) left_tile = prev_tile;
    const bool starts = act && tile != left_tile;
    const unsigned m = __ballot_sync(0xffffffffu, starts);
    const unsigned below = m & (0xffffffffu >> (31 - lane));
    const int start_k = below ? (k0 + 31 - __clz(below)) : prev_start;
    if (act) {
      const int64_t t = (int64_t)a.toff[((int64_t)hi * a.ntiles + tile) * a.NB + r] + (k - start_k);
      if (t < a.task_cap) {
        // a meta row is 24 bytes: three 8-byte stores (t * 24 is a multiple of 8)
        int2* mt = reinterpret_cast<int2*>(a.meta + t * MSA_TASK_META_COLS);
        mt[0] = make_int2(hi, r);
        mt[1] = make_int2(s, cnt);
        mt[2] = make_int2(d, b);
        int rows[kChunk], pos[kChunk];
        const int32_t* src = qi + s;
        if (cnt == kChunk && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
          const int4 x0 = reinterpret_cast<const int4*>(src)[0], x1 = reinterpret_cast<const int4*>(src)[1];
          pos[0] = x0.x; pos[1] = x0.y; pos[2] = x0.z; pos[3] = x0.w;
          pos[4] = x1.x; pos[5] = x1.y; pos[6] = x1.z; pos[7] = x1.w;
        } else {
#pragma unroll
          for (int i = 0; i < kChunk; ++i) pos[i] = i < cnt ? src[i] : -1;
        }
#pragma unroll
        for (int i = 0; i < kChunk; ++i) rows[i] = i < cnt ? tok0 + pos[i] : -1;
        int4* qr = reinterpret_cast<int4*>(a.q_rows + t * kChunk);
        int4* qp = reinterpret_cast<int4*>(a.q_pos + t * kChunk);
        qr[0] = make_int4(rows[0], rows[1], rows[2], rows[3]);
        qr[1] = make_int4(rows[4], rows[5], rows[6], rows[7]);
        qp[0] = make_int4(pos[0], pos[1], pos[2], pos[3]);
        qp[1] = make_int4(pos[4], pos[5], pos[6], pos[7]);
      }
    }
    const int last = min(31, ngroups - 1 - k0);
    prev_tile = __shfl_sync(0xffffffffu, tile, last);
    prev_start = __shfl_sync(0xffffffffu, start_k, last);
  }
}

// ---------------------------------------------------------------------------
// forward work plan: a stable counting sort of the (index head, chunk) items by
// selected-block count, longest first, items selecting nothing last
// ---------------------------------------------------------------------------
constexpr int kPlanBlock = 1024;         // items per block of the plan kernels
constexpr int kPlanBins = kMaxTopk + 1;  // selected-block counts 0 .. 32

struct PlanArgs {
  const int32_t* sel;
  const int32_t* cu;
  const int32_t* chunk_off;
  int32_t* hist;       // [nblk][kPlanBins]: counts, then exclusive output offsets
  int32_t* meta;       // [Hi * NC, 6]
  int32_t* work_count;
  int N, NC, K, Hi, nblk;
  int32_t* status;
};

// Bin of an item in output order: count K first, ..., count 1, then count 0.
__device__ __forceinline__ int plan_bin(int nsel, int K) { return nsel > 0 ? K - nsel : K; }

__device__ __forceinline__ int plan_nsel(const PlanArgs& a, int64_t item) {
  const int hi = (int)(item / a.NC), g = (int)(item % a.NC);
  int n = 0;
  const int32_t* row = a.sel + ((int64_t)hi * a.NC + g) * a.K;
  for (int k = 0; k < a.K; ++k) n += row[k] >= 0;
  return n;
}

__global__ void __launch_bounds__(kPlanBlock) plan_hist_kernel(PlanArgs a) {
  __shared__ int h[kPlanBins];
  if (status_bad(a.status)) return;
  if (threadIdx.x < kPlanBins) h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t item = (int64_t)blockIdx.x * kPlanBlock + threadIdx.x;
  if (item < (int64_t)a.Hi * a.NC) atomicAdd(&h[plan_bin(plan_nsel(a, item), a.K)], 1);
  __syncthreads();
  if (threadIdx.x < kPlanBins) a.hist[(int64_t)blockIdx.x * kPlanBins + threadIdx.x] = h[threadIdx.x];
}

// One block: output offset of every (block, bin) = items of earlier bins plus
// items of the same bin in earlier blocks; work_count = items of bins with a
// selected block.
__global__ void __launch_bounds__(1024) plan_scan_kernel(PlanArgs a) {
  __shared__ int ws[32];
  __shared__ int tot;
  if (status_bad(a.status)) return;
  int64_t carry = 0;
  for (int bin = 0; bin <= a.K; ++bin) {
    if (bin == a.K && threadIdx.x == 0) *a.work_count = (int32_t)carry;
    for (int base = 0; base < a.nblk; base += 1024) {
      const int b = base + threadIdx.x;
      const int v = b < a.nblk ? a.hist[(int64_t)b * kPlanBins + bin] : 0;
      const int e = block_excl_scan(v, ws, &tot);
      if (b < a.nblk) a.hist[(int64_t)b * kPlanBins + bin] = (int32_t)(carry + e);
      carry += tot;
    }
  }
}

// Each item's position: its block's offset for its bin plus its rank among the
// block's earlier items of the same bin (stable).
__global__ void __launch_bounds__(kPlanBlock) plan_scatter_kernel(PlanArgs a) {
  __shared__ int wcount[kPlanBlock / 32][kPlanBins];
  if (status_bad(a.status)) return;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kPlanBlock / 32) * kPlanBins; i += kPlanBlock) (&wcount[0][0])[i] = 0;
  __syncthreads();
  const int64_t item = (int64_t)blockIdx.x * kPlanBlock + threadIdx.x;
  const bool valid = item < (int64_t)a.Hi * a.NC;
  const int bin = valid ? plan_bin(plan_nsel(a, item), a.K) : kPlanBins;  // kPlanBins: no bin
  const unsigned same = __match_any_sync(0xffffffffu, bin);
  const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
  if (valid && rank_in_warp == 0) wcount[w][bin] = __popc(same);
  __syncthreads();
  if (!valid) return;
  int before = 0;
  for (int v = 0; v < w; ++v) before += wcount[v][bin];
  const int64_t pos = a.hist[(int64_t)blockIdx.x * kPlanBins + bin] + before + rank_in_warp;
  const int hi = (int)(item / a.NC), g = (int)(item % a.NC);
  const int d = upper_index(a.chunk_off, a.N + 1, g);
  const int c = g - a.chunk_off[d];
  const int len = a.cu[d + 1] - a.cu[d];
  int2* mt = reinterpret_cast<int2*>(a.meta + pos * MSA_TASK_META_COLS);
  mt[0] = make_int2(hi, g);
  mt[1] = make_int2(a.cu[d] + c * kChunk, min(kChunk, len - c * kChunk));
  mt[2] = make_int2(d, c * kChunk / kBlock);
}

size_t plan_ws_bytes(const msa_problem* p) {
  const int64_t items = (int64_t)p->num_index_heads * p->num_chunks, N = p->num_docs;
  const int64_t nblk = (items + kPlanBlock - 1) / kPlanBlock;
  return round_up(sizeof(int32_t) * 2 * (N + 1), 256) + round_up(sizeof(int32_t) * nblk * kPlanBins, 256);
}

// Scratch of msa_build_k2q_noalloc, for callers that may not allocate device
// memory.  Every device that loads the library holds one copy until exit.  In
// host code the name is only a host-side stand-in for the symbol, so the
// device address is looked up once per device and kept, together with the
// unique ID of the CUDA context it was looked up in: after cudaDeviceReset a
// new context (with the module loaded again, possibly elsewhere) gets a new
// ID, and the address is looked up again.
static __device__ __align__(256) uint8_t g_k2q_scratch[MSA_NOALLOC_SCRATCH_BYTES];

namespace {
struct ScratchAddr {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
ScratchAddr g_k2q_scratch_addr[kMaxDevices];
std::mutex g_k2q_scratch_mu;

// Unique ID of the calling thread's current CUDA context (driver entry points
// looked up through the runtime, so the library needs no link to libcuda).
int current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, id) != CUDA_SUCCESS)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

// Device address of g_k2q_scratch in the current device's current context.
int k2q_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MSA_ERR_INVALID_ARGUMENT;
  // No context may be current yet (the runtime binds the primary context on
  // its first real call): then the lookup below binds it, and its ID is read
  // after.
  unsigned long long ctx_id = 0;
  const bool have_ctx = current_context_id(&ctx_id) == MSA_OK;
  std::lock_guard<std::mutex> lk(g_k2q_scratch_mu);
  ScratchAddr& e = g_k2q_scratch_addr[dev];
  if (!have_ctx || !e.ptr || e.ctx_id != ctx_id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_k2q_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return MSA_ERR_CUDA;
    }
    if (!have_ctx && current_context_id(&ctx_id) != MSA_OK) return MSA_ERR_CUDA;
    e.ptr = ptr;
    e.ctx_id = ctx_id;
  }
  *out = e.ptr;
  return MSA_OK;
}
}  // namespace

}  // namespace msa

namespace msa {
int launch_layout(const msa_problem* p, int32_t* blk_off, int32_t* chunk_off, int32_t* status, cudaStream_t st) {
  layout_kernel<<<1, 1024, 0, st>>>(p->cu_seqlens, p->kv_doc_starts, p->num_docs, p->total_tokens, p->kv_rows,
                                    p->num_blocks, p->num_chunks, blk_off, chunk_off, status);
  return cuda_status(cudaGetLastError());
}
}  // namespace msa

using namespace msa;

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

const char* msa_status_string(int s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MSA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case MSA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MSA_ERR_CAPACITY: return "capacity too small";
    case MSA_ERR_INVALID_SELECTION: return "invalid key-block selection";
    case MSA_ERR_TIMEOUT: return "device wait timed out";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_INVALID_DOCUMENTS: return "inconsistent document offsets";
    case MSA_ERR_SCRATCH_TOO_SMALL: return "problem needs more scratch than the fixed no-allocation array holds";
    default: return "unknown status";
  }
}

int32_t msa_rows_per_cta(int64_t num_rows) { return num_rows < 2400 ? 4 : 64; }

void msa_chunk_map(int64_t n, int32_t R, int32_t S, int64_t* out3) {
  if (!out3 || R <= 0) return;
  const int64_t full = n / R, tail = n - full * R;
  out3[0] = full;
  out3[1] = tail;
  out3[2] = full + (tail < S ? tail : S);
}

int64_t msa_grid_launch_bound(int64_t cap, int32_t S) {
  // max over n in [0, cap] of full + min(tail, S).  In the small regime
  // (R = 4) tail < 4, in the large one (R = 64) tail < 64; the maximum of each
  // regime is at its largest n with the largest reachable tail.
  if (cap < 0 || S < 0) return 0;
  auto grid = [S](int64_t n) {
    const int64_t R = n < 2400 ? 4 : 64;
    const int64_t full = n / R, tail = n - full * R;
    return full + (tail < S ? tail : S);
  };
  int64_t best = 0;
  const int64_t small_hi = cap < 2399 ? cap : 2399;
  for (int64_t n = small_hi; n >= 0 && n > small_hi - 4; --n) best = best > grid(n) ? best : grid(n);
  if (cap >= 2400)
    for (int64_t n = cap; n >= 2400 && n > cap - 64; --n) best = best > grid(n) ? best : grid(n);
  return best;
}

int msa_device_capability(int32_t device, int32_t* major, int32_t* minor) {
  if (!major || !minor) return MSA_ERR_INVALID_ARGUMENT;
  msa::DevInfo d;
  int rc = msa::dev_info(device, &d);
  if (rc) return rc;
  *major = d.major;
  *minor = d.minor;
  return MSA_OK;
}

int msa_device_sm_count(int32_t device, int32_t* sms) {
  if (!sms) return MSA_ERR_INVALID_ARGUMENT;
  msa::DevInfo d;
  int rc = msa::dev_info(device, &d);
  if (rc) return rc;
  *sms = d.sms;
  return MSA_OK;
}

size_t msa_workspace_bytes(const msa_problem* p, int64_t edge_cap, int64_t task_cap, int32_t tile_chunks) {
  if (check_problem(p) != MSA_OK || edge_cap < 0 || task_cap < 0 || tile_chunks < 0) return 0;
  const size_t sizes[] = {k2q_ws_bytes(p), tasks_ws_bytes(p, tile_chunks), bwd_ws_bytes(p), select_ws_bytes(p),
                          plan_ws_bytes(p)};
  size_t m = 0;
  for (size_t x : sizes) m = x > m ? x : m;
  return m;
}

int msa_build_k2q(const msa_problem* p, const int32_t* sel, int32_t* row_ptr, int32_t* q_indices,
                  int64_t edge_cap, int32_t* d_status, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (!sel || !row_ptr || !q_indices || !d_status || !ws || edge_cap < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(sel) || !aligned16(row_ptr) || !aligned16(q_indices) || !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (edge_cap > INT32_MAX) return MSA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < k2q_ws_bytes(p)) return MSA_ERR_INVALID_ARGUMENT;
  if ((rc = check_device_current())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = p->num_docs, NB = p->num_blocks, NC = p->num_chunks, Hi = p->num_index_heads;
  K2QArgs a;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* blk_off = reinterpret_cast<int32_t*>(w);
  int32_t* chunk_off = blk_off + (N + 1);
  w += round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  const int64_t SG = k2q_group_chunks(NC), nS = (NC + SG - 1) / SG;
  a.cnt = reinterpret_cast<int32_t*>(w);
  w += round_up(sizeof(int32_t) * Hi * nS * NB, 256);
  a.totals = reinterpret_cast<int32_t*>(w);
  a.sel = sel; a.cu = p->cu_seqlens; a.blk_off = blk_off; a.chunk_off = chunk_off;
  a.row_ptr = row_ptr; a.q_indices = q_indices; a.edge_cap = edge_cap;
  a.N = N; a.NB = NB; a.NC = NC; a.K = p->topk; a.SG = (int)SG; a.nS = (int)nS; a.status = d_status;

  layout_kernel<<<1, 1024, 0, st>>>(p->cu_seqlens, p->kv_doc_starts, N, p->total_tokens, p->kv_rows, NB, NC,
                                    blk_off, chunk_off, d_status);
  const size_t hist_bytes = sizeof(int) * NB;
  if (hist_bytes > 48 * 1024) {
    if ((rc = cuda_status(cudaFuncSetAttribute(k2q_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)hist_bytes))) ||
        (rc = cuda_status(cudaFuncSetAttribute(k2q_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)hist_bytes))))
      return rc;
  }
  k2q_count_kernel<<<dim3((unsigned)nS, Hi), 256, hist_bytes, st>>>(a);
  const int64_t rows = (int64_t)Hi * NB;
  k2q_group_offsets_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, st>>>(a, Hi);
  k2q_row_ptr_kernel<<<Hi, 1024, 0, st>>>(a);
  k2q_scatter_kernel<<<dim3((unsigned)nS, Hi), 32, hist_bytes, st>>>(a);
  return cuda_status(cudaGetLastError());
}

// Same build as msa_build_k2q with g_k2q_scratch as its workspace.
int msa_build_k2q_noalloc(const msa_problem* p, const int32_t* sel, int32_t* row_ptr, int32_t* q_indices,
                          int64_t edge_cap, int32_t* d_status, void* stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (k2q_ws_bytes(p) > MSA_NOALLOC_SCRATCH_BYTES) return MSA_ERR_SCRATCH_TOO_SMALL;
  if ((rc = check_device_current())) return rc;
  void* scratch = nullptr;
  if ((rc = k2q_scratch_address(&scratch))) return rc;
  return msa_build_k2q(p, sel, row_ptr, q_indices, edge_cap, d_status, scratch, MSA_NOALLOC_SCRATCH_BYTES, stream);
}

int msa_build_tasks(const msa_problem* p, const int32_t* row_ptr, const int32_t* q_indices, int64_t edge_cap,
                    int32_t tile_chunks, int32_t* task_meta, int32_t* task_q_rows, int32_t* task_q_pos,
                    int32_t* walk, int64_t task_cap, int32_t num_sms, int32_t* d_status, void* ws,
                    size_t ws_bytes, void* stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (!row_ptr || !q_indices || !task_meta || !task_q_rows || !task_q_pos || !walk || !d_status || !ws)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(row_ptr) || !aligned16(q_indices) || !aligned16(task_meta) || !aligned16(task_q_rows) ||
      !aligned16(task_q_pos) || !aligned16(walk) || !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (edge_cap < 1 || edge_cap > INT32_MAX || task_cap < 1 || task_cap > INT32_MAX || tile_chunks < 0 ||
      num_sms < 0)
    return MSA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < tasks_ws_bytes(p, tile_chunks)) return MSA_ERR_INVALID_ARGUMENT;
  if ((rc = check_device_current())) return rc;
  if (num_sms == 0 && (rc = sm_count_current(&num_sms))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = p->num_docs, NB = p->num_blocks, NC = p->num_chunks, Hi = p->num_index_heads;
  const int64_t ntiles = num_tiles(NC, tile_chunks);
  const int64_t n = (int64_t)Hi * ntiles * NB;
  if (n > INT32_MAX) return MSA_ERR_UNSUPPORTED_SHAPE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  TaskArgs a;
  int32_t* blk_off = reinterpret_cast<int32_t*>(w);
  int32_t* chunk_off = blk_off + (N + 1);
  w += round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  a.tcnt = reinterpret_cast<int32_t*>(w);
  w += round_up(sizeof(int32_t) * n, 256);
  a.toff = reinterpret_cast<int32_t*>(w);
  w += round_up(sizeof(int32_t) * n, 256);
  a.bsum = reinterpret_cast<int32_t*>(w);
  a.row_ptr = row_ptr; a.q_indices = q_indices; a.cu = p->cu_seqlens; a.blk_off = blk_off;
  a.chunk_off = chunk_off; a.meta = task_meta; a.q_rows = task_q_rows; a.q_pos = task_q_pos; a.walk = walk;
  a.edge_cap = edge_cap; a.task_cap = task_cap; a.N = N; a.NB = NB; a.NC = NC; a.Hi = Hi;
  a.tile_chunks = tile_chunks; a.ntiles = (int)ntiles; a.num_sms = num_sms; a.status = d_status;

  layout_kernel<<<1, 1024, 0, st>>>(p->cu_seqlens, p->kv_doc_starts, N, p->total_tokens, p->kv_rows, NB, NC,
                                    blk_off, chunk_off, d_status);
  if ((rc = cuda_status(cudaMemsetAsync(a.tcnt, 0, sizeof(int32_t) * n, st)))) return rc;
  const int64_t warps = (int64_t)Hi * NB;
  const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
  task_count_kernel<<<blocks, 256, 0, st>>>(a);
  const int nblk = (int)((n + kScanSeg - 1) / kScanSeg);
  scan_reduce_kernel<<<nblk, 1024, 0, st>>>(a.tcnt, n, a.bsum, d_status);
  scan_bsums_walk_kernel<<<1, 1024, 0, st>>>(a.bsum, nblk, a);
  scan_apply_kernel<<<nblk, 1024, 0, st>>>(a.tcnt, n, a.bsum, a.toff, d_status);
  task_emit_kernel<<<blocks, 256, 0, st>>>(a);
  return cuda_status(cudaGetLastError());
}

int msa_plan_forward(const msa_problem* p, const int32_t* sel, int32_t* scheduler_metadata, int32_t* work_count,
                     int32_t* d_status, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (!sel || !scheduler_metadata || !work_count || !d_status || !ws) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(sel) || !aligned16(scheduler_metadata) || !aligned16(work_count) || !aligned16(d_status) ||
      !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < plan_ws_bytes(p)) return MSA_ERR_INVALID_ARGUMENT;
  if ((rc = check_device_current())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = p->num_docs;
  const int64_t items = (int64_t)p->num_index_heads * p->num_chunks;
  if (items > INT32_MAX / 2) return MSA_ERR_UNSUPPORTED_SHAPE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* blk_off = reinterpret_cast<int32_t*>(w);
  int32_t* chunk_off = blk_off + (N + 1);
  w += round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  PlanArgs a;
  a.sel = sel; a.cu = p->cu_seqlens; a.chunk_off = chunk_off; a.hist = reinterpret_cast<int32_t*>(w);
  a.meta = scheduler_metadata; a.work_count = work_count; a.N = N; a.NC = p->num_chunks; a.K = p->topk;
  a.Hi = p->num_index_heads; a.nblk = (int)((items + kPlanBlock - 1) / kPlanBlock); a.status = d_status;
  if ((rc = launch_layout(p, blk_off, chunk_off, d_status, st))) return rc;
  plan_hist_kernel<<<a.nblk, kPlanBlock, 0, st>>>(a);
  plan_scan_kernel<<<1, 1024, 0, st>>>(a);
  plan_scatter_kernel<<<a.nblk, kPlanBlock, 0, st>>>(a);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Self-test of the bounded waits: an mbarrier phase that nothing completes.
// ---------------------------------------------------------------------------
namespace msa {
__global__ void selftest_wait_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // no thread ever arrives: the wait gives up after kWaitLimitNs and records
  // MSA_ERR_TIMEOUT in *status
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, status);
}
}  // namespace msa

extern "C" int msa_selftest_wait_timeout(int32_t* d_status, void* stream) {
  if (!d_status || !msa::aligned16(d_status)) return MSA_ERR_INVALID_ARGUMENT;
  int rc = msa::check_device_current();
  if (rc) return rc;
  msa::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d_status);
  return msa::cuda_status(cudaGetLastError());
}
