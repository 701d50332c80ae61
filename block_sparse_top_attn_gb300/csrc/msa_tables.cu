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
  if (p->head_dim != kHeadDim || (p->block_size != 64 && p->block_size != 128) || p->query_chunk != kChunk)
    return MSA_ERR_UNSUPPORTED_SHAPE;
  if (p->num_kv_heads != p->num_index_heads || p->num_q_heads != kGroup * p->num_index_heads)
    return MSA_ERR_UNSUPPORTED_SHAPE;
  if (p->topk < 1 || p->topk > kMaxTopk) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (p->num_blocks < 1 || p->num_chunks < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (p->num_blocks > kMaxRows) return MSA_ERR_UNSUPPORTED_SHAPE;
  // counts implied by T alone bound the per-document sums
  const int64_t T = p->total_tokens, N = p->num_docs;
  if (p->num_chunks < (T + kChunk - 1) / kChunk || p->num_chunks > T / kChunk + N) return MSA_ERR_INVALID_ARGUMENT;
  const int64_t B = p->block_size;
  if (p->num_blocks < (T + B - 1) / B || p->num_blocks > T / B + N) return MSA_ERR_INVALID_ARGUMENT;
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
  const int64_t n = Hi * num_tiles(NC, tile_chunks) * NB * key_tiles_per_block(p);
  size_t b = round_up(sizeof(int32_t) * 2 * (N + 1), 256);
  b += round_up(sizeof(int32_t) * n, 256) * 2;
  b += round_up(sizeof(int32_t) * ((n + kScanSeg - 1) / kScanSeg + 1), 256);
  return b;
}

size_t bwd_ws_bytes(const msa_problem* p, bool dq_fp32) {
  const int64_t T = p->total_tokens, Hq = p->num_q_heads, W = p->kv_rows, Hkv = p->num_kv_heads;
  size_t b = round_up(sizeof(float) * T * Hq, 256);                 // D
  b += 2 * round_up(sizeof(float) * W * Hkv * kHeadDim, 256);       // dK, dV accumulators
  b += 256;                                                          // walk-unit counter
  if (dq_fp32) b += round_up(sizeof(float) * T * Hq * kHeadDim, 256);  // fp32 dQ accumulator
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
                                                       int B, int NB, int NC, int32_t* blk_off, int32_t* chunk_off,
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
      nb = len > 0 ? (len + B - 1) / B : 0;
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
// The selection is cut into scatter groups of SG consecutive query chunks.
// Pass 1 counts, per (index head, group), the entries each key-block row
// receives; pass 2 turns the counts into each group's offset inside each row
// and the row totals; pass 3 scans the totals into row_ptr; pass 4 places
// each group's entries and writes them.  Passes 1 and 4 stage the group's
// selection in shared memory 64 chunks at a time, take the staged chunks 32
// (a piece) at a time, and keep, per row, a 32-bit mask of the piece's
// chunks that selected it.  An entry's place in
// its row follows from the mask: the row's cursor plus 8 for every earlier
// chunk of the piece in the mask (only a document's last chunk can hold fewer
// than 8 queries, and no later chunk of its document selects anything), so
// the order of positions within a row needs no sequential walk.  Rows are
// handled in windows of at most win rows per pass, which bounds the shared
// memory.
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
  int N, NB, NC, K, SG, nS, B;
  int win;            // rows per window of passes 1 and 4
  int32_t* status;
};

constexpr int kPiece = 32;          // query chunks placed at a time: one mask bit each
constexpr int kStage = 64;          // query chunks staged at a time (two pieces)
constexpr int kRowWindow = 16384;   // largest row window of passes 1 and 4

// The staged chunks of a group: per chunk its first position, its query
// count, its document's first row relative to the group's first row, its
// document's block count, and its selection slots.
constexpr int kSelStride = kMaxTopk + 1;  // a staged chunk's slots (padded: a lane per chunk reads conflict-free)
struct K2QStage {
  int v0[kStage];
  int len[kStage];
  int rbase[kStage];
  int nbd[kStage];
  int sel[kStage * kSelStride];  // slots K .. 31 hold -1
};
static_assert(sizeof(K2QStage) % 16 == 0, "the stage keeps 16-byte alignment of what follows");

// Rows [r_lo, r_hi) of the documents that group s's chunks belong to.
__device__ __forceinline__ void group_rows(const K2QArgs& a, int s, int* r_lo, int* r_hi) {
  const int g0 = s * a.SG;
  const int g1 = min(a.NC, g0 + a.SG) - 1;
  const int d0 = upper_index(a.chunk_off, a.N + 1, g0);
  const int d1 = upper_index(a.chunk_off, a.N + 1, g1);
  *r_lo = a.blk_off[d0];
  *r_hi = a.blk_off[d1 + 1];
}

// All threads of the block: stage chunks [g0, g0 + nc) of index head hi.  The
// selection rows go by asynchronous 4-byte copies, a warp per chunk row, all
// in flight at once while the threads look up each chunk's document.
__device__ __forceinline__ void stage_chunks(const K2QArgs& a, int hi, int g0, int nc, int r_lo, K2QStage& S) {
  const int32_t* src = a.sel + ((int64_t)hi * a.NC + g0) * a.K;
  const int lane = threadIdx.x & 31;
  for (int j = threadIdx.x >> 5; j < nc; j += blockDim.x >> 5) {
    int* dst = &S.sel[j * kSelStride + lane];
    if (lane < a.K)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src + j * a.K + lane)
                   : "memory");
    else
      *dst = -1;
  }
  for (int j = threadIdx.x; j < nc; j += blockDim.x) {
    const int g = g0 + j;
    const int d = upper_index(a.chunk_off, a.N + 1, g);
    const int c = g - a.chunk_off[d];
    S.v0[j] = c * kChunk;
    S.len[j] = min(kChunk, a.cu[d + 1] - a.cu[d] - c * kChunk);
    S.rbase[j] = a.blk_off[d] - r_lo;
    S.nbd[j] = a.blk_off[d + 1] - a.blk_off[d];
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Pass 1, per (scatter group, index head): validate the selection and count
// query entries per key-block row.  A lane per staged chunk and, per warp,
// every 8th slot; a slot that sets a mask bit its own chunk already set is a
// duplicate.
constexpr int kCountThreads = 256;
constexpr int kCountSlots = kMaxTopk / (kCountThreads / 32);  // slots per thread

__global__ void __launch_bounds__(kCountThreads) k2q_count_kernel(K2QArgs a) {
  extern __shared__ __align__(16) int k2q_smem[];
  K2QStage& S = *reinterpret_cast<K2QStage*>(k2q_smem);
  int* hist = k2q_smem + sizeof(K2QStage) / sizeof(int);
  uint32_t* mask = reinterpret_cast<uint32_t*>(hist + a.win);
  if (status_bad(a.status)) return;
  const int s = blockIdx.x, hi = blockIdx.y;
  const int j = threadIdx.x & 31, w = threadIdx.x >> 5;
  int r_lo, r_hi;
  group_rows(a, s, &r_lo, &r_hi);
  int32_t* out = a.cnt + ((int64_t)hi * a.nS + s) * a.NB;
  for (int r = threadIdx.x; r < a.NB; r += blockDim.x)
    if (r < r_lo || r >= r_hi) out[r] = 0;
  const int g_begin = s * a.SG, g_end = min(a.NC, g_begin + a.SG);
  const uint32_t bit = 1u << j;
  for (int w0 = r_lo; w0 < r_hi; w0 += a.win) {
    const int w1 = min(r_hi, w0 + a.win);
    __syncthreads();  // the previous window's counts are written out
    for (int i = threadIdx.x; i < w1 - w0; i += blockDim.x) {
      hist[i] = 0;
      mask[i] = 0;
    }
    for (int gs = g_begin; gs < g_end; gs += kStage) {
      const int nc = min(kStage, g_end - gs);
      __syncthreads();  // the previous stage is consumed
      stage_chunks(a, hi, gs, nc, r_lo, S);
      __syncthreads();
      for (int pc = 0; pc < nc; pc += kPiece) {
        const int c = pc + j;  // this lane's staged chunk
        const bool jv = c < nc;
        const int len = jv ? S.len[c] : 0, v0 = jv ? S.v0[c] : 0, nbd = jv ? S.nbd[c] : 0;
        const int rb = jv ? r_lo + S.rbase[c] - w0 : 0;
        int x[kCountSlots];  // row - w0 of each of this thread's entries, or -1
#pragma unroll
        for (int i = 0; i < kCountSlots; ++i) {
          x[i] = -1;
          const int b = jv ? S.sel[c * kSelStride + w + (kCountThreads / 32) * i] : -1;
          if (b == -1) continue;
          if (b < 0 || b >= nbd || (int64_t)b * a.B > v0) {
            set_status(a.status, MSA_ERR_INVALID_SELECTION);
            continue;
          }
          const int xr = rb + b;
          if (xr < 0 || xr >= w1 - w0) continue;
          x[i] = xr;
          if (atomicOr(&mask[xr], bit) & bit) set_status(a.status, MSA_ERR_INVALID_SELECTION);
          atomicAdd(&hist[xr], len);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kCountSlots; ++i)
          if (x[i] >= 0) mask[x[i]] = 0;
        __syncthreads();  // masks clear for the next piece
      }
    }
    __syncthreads();
    for (int r = w0 + (int)threadIdx.x; r < w1; r += blockDim.x) out[r] = hist[r - w0];
  }
}

// Pass 2, a block per (32 rows, index head): each warp sums a contiguous
// range of groups for the block's 32 rows (a lane per row, coalesced), the
// ranges are scanned across warps, and each warp writes its groups' exclusive
// offsets.  The row totals go to totals.
__global__ void __launch_bounds__(1024) k2q_group_offsets_kernel(K2QArgs a) {
  __shared__ int part[32][33];
  if (status_bad(a.status)) return;
  const int hi = blockIdx.y, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int r = blockIdx.x * 32 + lane;
  const bool ok = r < a.NB;
  const int per = (a.nS + 31) / 32;
  const int s0 = min(a.nS, w * per), s1 = min(a.nS, s0 + per);
  int32_t* col = a.cnt + (int64_t)hi * a.nS * a.NB + r;
  int sum = 0;
  if (ok)
    for (int s = s0; s < s1; ++s) sum += col[(int64_t)s * a.NB];
  part[w][lane] = sum;
  __syncthreads();
  if (w == 0) {
    int run = 0;
    for (int i = 0; i < 32; ++i) {
      const int v = part[i][lane];
      part[i][lane] = run;
      run += v;
    }
    if (ok) a.totals[(int64_t)hi * a.NB + r] = run;
  }
  __syncthreads();
  if (ok) {
    int run = part[w][lane];
    for (int s = s0; s < s1; ++s) {
      int32_t* c = col + (int64_t)s * a.NB;
      const int v = *c;
      *c = run;
      run += v;
    }
  }
}

// Pass 3, per index head: row_ptr = exclusive scan of the row totals.
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

constexpr int kScatterThreads = 128;

// Eight consecutive ints v0 .. v0+7 at a 32-byte aligned address: one 256-bit store.
__device__ __forceinline__ void st_global_iota8(int32_t* dst, int v0) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v0), "r"(v0 + 1),
               "r"(v0 + 2), "r"(v0 + 3), "r"(v0 + 4), "r"(v0 + 5), "r"(v0 + 6), "r"(v0 + 7)
               : "memory");
}

// Pass 4, per (scatter group, index head), one row window at a time: for each
// staged piece, mark every (chunk, slot) in its row's mask; place each entry at
// the row's cursor plus 8 per earlier marked chunk; let the row's first chunk
// advance the cursor past the piece and clear the mask; write the entries.  A
// lane per chunk and, per warp, every 4th slot, so the lanes of a warp write
// one slot of consecutive chunks (chunks that selected the same row, a
// block's chunks and their diagonal or recent blocks, write neighbouring
// entries together).
constexpr int kScatterSlots = kMaxTopk / (kScatterThreads / 32);  // slots per thread

__global__ void __launch_bounds__(kScatterThreads) k2q_scatter_kernel(K2QArgs a) {
  extern __shared__ __align__(16) int k2q_smem[];
  K2QStage& S = *reinterpret_cast<K2QStage*>(k2q_smem);
  int* cursor = k2q_smem + sizeof(K2QStage) / sizeof(int);
  uint32_t* mask = reinterpret_cast<uint32_t*>(cursor + a.win);
  if (status_bad(a.status)) return;
  const int s = blockIdx.x, hi = blockIdx.y;
  const int j = threadIdx.x & 31, w = threadIdx.x >> 5;
  int r_lo, r_hi;
  group_rows(a, s, &r_lo, &r_hi);
  const int32_t* rp = a.row_ptr + (int64_t)hi * (a.NB + 1);
  const int32_t* off = a.cnt + ((int64_t)hi * a.nS + s) * a.NB;
  int32_t* qi = a.q_indices + (int64_t)hi * a.edge_cap;
  const int g_begin = s * a.SG, g_end = min(a.NC, g_begin + a.SG);
  const uint32_t bit = 1u << j, below = bit - 1u;
  for (int w0 = r_lo; w0 < r_hi; w0 += a.win) {
    const int w1 = min(r_hi, w0 + a.win);
    __syncthreads();  // the previous window's pieces are written
#pragma unroll 4
    for (int r = w0 + (int)threadIdx.x; r < w1; r += blockDim.x) {
      cursor[r - w0] = rp[r] + off[r];
      mask[r - w0] = 0;
    }
    for (int gs = g_begin; gs < g_end; gs += kStage) {
      const int nc = min(kStage, g_end - gs);
      __syncthreads();  // cursors ready; the previous stage is consumed
      stage_chunks(a, hi, gs, nc, r_lo, S);
      __syncthreads();
      for (int pc = 0; pc < nc; pc += kPiece) {
        const int c = pc + j;  // this lane's staged chunk
        const bool jv = c < nc;
        const int len = jv ? S.len[c] : 0, v0 = jv ? S.v0[c] : 0;
        const int rb = jv ? r_lo + S.rbase[c] - w0 : 0;
        int x[kScatterSlots];  // row - w0 of each of this thread's entries, or -1
#pragma unroll
        for (int i = 0; i < kScatterSlots; ++i) {
          const int b = jv ? S.sel[c * kSelStride + w + (kScatterThreads / 32) * i] : -1;
          const int xr = rb + b;
          x[i] = (b >= 0 && xr >= 0 && xr < w1 - w0) ? xr : -1;
          if (x[i] >= 0) atomicOr(&mask[x[i]], bit);
        }
        __syncthreads();
        int p[kScatterSlots], adv[kScatterSlots];
#pragma unroll
        for (int i = 0; i < kScatterSlots; ++i) {
          p[i] = -1;
          adv[i] = -1;
          if (x[i] < 0) continue;
          const uint32_t m = mask[x[i]];
          p[i] = cursor[x[i]] + kChunk * __popc(m & below);
          if ((m & below) == 0)  // the row's first chunk in this piece
            adv[i] = kChunk * (__popc(m) - 1) + S.len[pc + 31 - __clz(m)];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kScatterSlots; ++i) {
          if (adv[i] >= 0) {
            cursor[x[i]] += adv[i];
            mask[x[i]] = 0;
          }
          if (p[i] < 0 || (int64_t)p[i] + len > a.edge_cap) continue;
          int32_t* dst = qi + p[i];
          const uintptr_t addr = reinterpret_cast<uintptr_t>(dst);
          if (len == kChunk && (addr & 31) == 0) {
            st_global_iota8(dst, v0);
          } else if (len == kChunk && (addr & 15) == 0) {
            reinterpret_cast<int4*>(dst)[0] = make_int4(v0, v0 + 1, v0 + 2, v0 + 3);
            reinterpret_cast<int4*>(dst)[1] = make_int4(v0 + 4, v0 + 5, v0 + 6, v0 + 7);
          } else {
            for (int e = 0; e < len; ++e) dst[e] = v0 + e;
          }
        }
        __syncthreads();  // cursors advanced, masks clear for the next piece
      }
    }
  }
}

// ---------------------------------------------------------------------------
// task build
// ---------------------------------------------------------------------------
// A task is one group of up to 8 consecutive CSR entries (one query chunk)
// against one 64-key tile of its row's block.  With 64-key blocks that is the
// block itself; a 128-key block gives up to two tasks per group, one per
// 64-key half, the upper half only when the group's last query reaches it.
// Task rows live in a key-tile row space: row r, half h -> rt = r * nh + h.
// Tasks are ordered by (index head, query tile, rt, CSR offset), so the
// tasks sharing a K/V tile are consecutive.
struct TaskArgs {
  const int32_t* row_ptr;
  const int32_t* q_indices;
  const int32_t* cu;
  const int32_t* blk_off;
  const int32_t* chunk_off;
  int32_t* tcnt;   // [Hi][ntiles][NBt] task counts
  int32_t* toff;   // exclusive scan of tcnt
  int32_t* bsum;   // per scan block sums
  int32_t* meta;
  int32_t* q_rows;
  int32_t* q_pos;
  int32_t* walk;
  int64_t edge_cap, task_cap;
  int N, NB, NBt, NC, Hi, tile_chunks, ntiles, num_sms, B, nh;
  int32_t* status;
};

// Warps per CSR row in the count and emit passes: warp p of a row takes the
// row's 32-group slabs p, p + kRowParts, ..., so long rows spread over
// kRowParts warps.
constexpr int kRowParts = 4;

__device__ __forceinline__ int task_tile(const TaskArgs& a, int64_t g) {
  return a.tile_chunks > 0 ? (int)(g / a.tile_chunks) : 0;
}

__device__ __forceinline__ int64_t tcnt_index(const TaskArgs& a, int hi, int tile, int rt) {
  return ((int64_t)hi * a.ntiles + tile) * a.NBt + rt;
}

// The (index head, row, part) of the calling warp; false past the last row.
__device__ __forceinline__ bool task_warp(const TaskArgs& a, int* hi, int* r, int* part) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (int64_t)a.Hi * a.NB * kRowParts) return false;
  *part = (int)(wid % kRowParts);
  const int64_t hr = wid / kRowParts;
  *hi = (int)(hr / a.NB);
  *r = (int)(hr % a.NB);
  return true;
}

// Count the row's tasks per query tile and key tile: tcnt[hi][tile][rt].
// Runs of equal tiles within a slab are added once.
__global__ void __launch_bounds__(256) task_count_kernel(TaskArgs a) {
  if (status_bad(a.status)) return;
  int hi, r, part;
  if (!task_warp(a, &hi, &r, &part)) return;
  const int lane = threadIdx.x & 31;
  const int32_t* rp = a.row_ptr + (int64_t)hi * (a.NB + 1);
  const int lo = rp[r], end = rp[r + 1];
  if (lo < 0 || end < lo || end > a.edge_cap) {
    if (lane == 0) set_status(a.status, MSA_ERR_INVALID_ARGUMENT);
    return;
  }
  const int ngroups = (end - lo + kChunk - 1) / kChunk;
  if (part * 32 >= ngroups) return;
  const int d = upper_index(a.blk_off, a.N + 1, r);
  const int len_d = a.cu[d + 1] - a.cu[d];
  const int upper_key0 = (r - a.blk_off[d]) * a.B + kKeyTile;  // first key of the upper half
  const int32_t* qi = a.q_indices + (int64_t)hi * a.edge_cap;
  for (int k0 = part * 32; k0 < ngroups; k0 += 32 * kRowParts) {
    const int k = k0 + lane;
    int tile = -1;
    bool upper = false;
    if (k < ngroups) {
      const int s = lo + k * kChunk;
      const int cnt = min(kChunk, end - s);
      const int pos = qi[s], last = qi[s + cnt - 1];
      if (pos < 0 || last >= len_d || last < pos) {
        set_status(a.status, MSA_ERR_INVALID_ARGUMENT);
      } else {
        tile = task_tile(a, (int64_t)a.chunk_off[d] + pos / kChunk);
        upper = a.nh > 1 && last >= upper_key0;
      }
    }
    // The lanes counted for a key tile are consecutive (all valid groups for
    // the lower tile, a suffix of them for the upper one) and their query
    // tiles ascend, so equal tiles form runs: the first lane of each run adds
    // the run's length.
    for (int h = 0; h < a.nh; ++h) {
      const int key = (tile >= 0 && (h == 0 || upper)) ? tile : -1;
      const int left = __shfl_up_sync(0xffffffffu, key, 1);
      const bool start = key >= 0 && (lane == 0 || left != key);
      const unsigned starts = __ballot_sync(0xffffffffu, start);
      const unsigned valid = __ballot_sync(0xffffffffu, key >= 0);
      if (start) {
        const unsigned after = lane == 31 ? 0u : (starts >> (lane + 1)) << (lane + 1);
        const int end = after ? __ffs(after) - 1 : 32 - __clz(valid);
        atomicAdd(&a.tcnt[tcnt_index(a, hi, key, r * a.nh + h)], end - lane);
      }
    }
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

// 256-bit global load / store of 8 ints (32-byte aligned addresses).
__device__ __forceinline__ void ld_global_v8(const int32_t* src, int (&v)[8]) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(src));
}
__device__ __forceinline__ void st_global_v8(int32_t* dst, const int (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Writes one task: its meta row and its 8 query rows and positions.
__device__ __forceinline__ void write_task(const TaskArgs& a, int64_t t, int hi, int rt, int s, int cnt, int d,
                                          int kb, int tok0, const int (&pos)[kChunk]) {
  // a meta row is 24 bytes: three 8-byte stores (t * 24 is a multiple of 8)
  int2* mt = reinterpret_cast<int2*>(a.meta + t * MSA_TASK_META_COLS);
  mt[0] = make_int2(hi, rt);
  mt[1] = make_int2(s, cnt);
  mt[2] = make_int2(d, kb);
  int rows[kChunk];
#pragma unroll
  for (int i = 0; i < kChunk; ++i) rows[i] = pos[i] >= 0 ? tok0 + pos[i] : -1;
  int32_t* qr = a.q_rows + t * kChunk;
  int32_t* qp = a.q_pos + t * kChunk;
  if (((reinterpret_cast<uintptr_t>(qr) | reinterpret_cast<uintptr_t>(qp)) & 31) == 0) {
    st_global_v8(qr, rows);
    st_global_v8(qp, pos);
  } else {  // 16-byte aligned (the ABI's minimum)
    reinterpret_cast<int4*>(qr)[0] = make_int4(rows[0], rows[1], rows[2], rows[3]);
    reinterpret_cast<int4*>(qr)[1] = make_int4(rows[4], rows[5], rows[6], rows[7]);
    reinterpret_cast<int4*>(qp)[0] = make_int4(pos[0], pos[1], pos[2], pos[3]);
    reinterpret_cast<int4*>(qp)[1] = make_int4(pos[4], pos[5], pos[6], pos[7]);
  }
}

// Emit the row's tasks.  A group's task index is the scan offset of its
// (query tile, key tile) plus its rank among the row's groups of that tile
// that reach the key tile.  The groups of a row are in ascending position, so
// its tiles ascend with the group index: the rank is the group index minus the
// first group of the tile (the tile prefix of the row's counts), and for the
// upper half also minus the groups before the first that reaches it (they
// are a prefix of the row).
__global__ void __launch_bounds__(256) task_emit_kernel(TaskArgs a) {
  if (status_bad(a.status)) return;
  int hi, r, part;
  if (!task_warp(a, &hi, &r, &part)) return;
  const int lane = threadIdx.x & 31;
  const int32_t* rp = a.row_ptr + (int64_t)hi * (a.NB + 1);
  const int lo = rp[r], end = rp[r + 1];
  const int ngroups = (end - lo + kChunk - 1) / kChunk;
  if (part * 32 >= ngroups) return;
  const int d = upper_index(a.blk_off, a.N + 1, r);
  const int b = r - a.blk_off[d];
  const int tok0 = a.cu[d];
  const int upper_key0 = b * a.B + kKeyTile;
  const int32_t* qi = a.q_indices + (int64_t)hi * a.edge_cap;
  // Tile tables, lane t for tile t when there are at most 32 tiles: the
  // row's first group in tile t, and the scan offsets of (t, rt) per half.
  const bool small = a.ntiles <= 32;
  int first_k = 0, off0 = 0, off1 = 0;
  if (small) {
    const int t = lane;
    const int c0 = t < a.ntiles ? a.tcnt[tcnt_index(a, hi, t, r * a.nh)] : 0;
    int x = c0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    first_k = x - c0;
    if (t < a.ntiles) {
      off0 = a.toff[tcnt_index(a, hi, t, r * a.nh)];
      if (a.nh > 1) off1 = a.toff[tcnt_index(a, hi, t, r * a.nh + 1)];
    }
  }
  // Groups that stop short of the upper half: a prefix of the row, at most
  // the 8 chunks that start inside the lower half.
  int n_short = 0;
  if (a.nh > 1) {
    const int k = lane;
    bool short_k = false;
    if (k < ngroups) {
      const int s = lo + k * kChunk;
      short_k = qi[min(s + kChunk, end) - 1] < upper_key0;
    }
    n_short = __popc(__ballot_sync(0xffffffffu, short_k));
  }
  for (int k0 = part * 32; k0 < ngroups; k0 += 32 * kRowParts) {
    const int k = k0 + lane;
    const bool act = k < ngroups;
    int s = 0, cnt = 0, tile = 0;
    int pos[kChunk];
    if (act) {
      s = lo + k * kChunk;
      cnt = min(kChunk, end - s);
      const int32_t* src = qi + s;
      if (cnt == kChunk && (reinterpret_cast<uintptr_t>(src) & 31) == 0) {
        ld_global_v8(src, pos);
      } else if (cnt == kChunk && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const int4 x0 = reinterpret_cast<const int4*>(src)[0], x1 = reinterpret_cast<const int4*>(src)[1];
        pos[0] = x0.x; pos[1] = x0.y; pos[2] = x0.z; pos[3] = x0.w;
        pos[4] = x1.x; pos[5] = x1.y; pos[6] = x1.z; pos[7] = x1.w;
      } else {
#pragma unroll
        for (int i = 0; i < kChunk; ++i) pos[i] = i < cnt ? src[i] : -1;
      }
      tile = task_tile(a, (int64_t)a.chunk_off[d] + pos[0] / kChunk);
    }
    int fk, o0, o1;
    if (small) {
      fk = __shfl_sync(0xffffffffu, first_k, tile);
      o0 = __shfl_sync(0xffffffffu, off0, tile);
      o1 = __shfl_sync(0xffffffffu, off1, tile);
    } else {
      fk = 0;
      for (int t2 = 0; act && t2 < tile; ++t2) fk += a.tcnt[tcnt_index(a, hi, t2, r * a.nh)];
      o0 = act ? a.toff[tcnt_index(a, hi, tile, r * a.nh)] : 0;
      o1 = act && a.nh > 1 ? a.toff[tcnt_index(a, hi, tile, r * a.nh + 1)] : 0;
    }
    if (!act) continue;
    const int64_t t0 = (int64_t)o0 + (k - fk);
    if (t0 < a.task_cap) write_task(a, t0, hi, r * a.nh, s, cnt, d, b * a.nh, tok0, pos);
    if (a.nh > 1 && k >= n_short) {
      const int64_t t1 = (int64_t)o1 + (k - max(fk, n_short));
      if (t1 < a.task_cap) write_task(a, t1, hi, r * a.nh + 1, s, cnt, d, b * a.nh + 1, tok0, pos);
    }
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
  int N, NC, K, Hi, nblk, B;
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
  mt[2] = make_int2(d, c * kChunk / a.B);
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
                                    p->block_size, p->num_blocks, p->num_chunks, blk_off, chunk_off, status);
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

size_t msa_workspace_bytes_opts(const msa_problem* p, int64_t edge_cap, int64_t task_cap, int32_t tile_chunks,
                                uint32_t options) {
  if (check_problem(p) != MSA_OK || edge_cap < 0 || task_cap < 0 || tile_chunks < 0) return 0;
  if (options & ~(uint32_t)MSA_BWD_DQ_FP32) return 0;
  const size_t sizes[] = {k2q_ws_bytes(p), tasks_ws_bytes(p, tile_chunks),
                          bwd_ws_bytes(p, (options & MSA_BWD_DQ_FP32) != 0), select_ws_bytes(p), plan_ws_bytes(p)};
  size_t m = 0;
  for (size_t x : sizes) m = x > m ? x : m;
  return m;
}

size_t msa_workspace_bytes(const msa_problem* p, int64_t edge_cap, int64_t task_cap, int32_t tile_chunks) {
  return msa_workspace_bytes_opts(p, edge_cap, task_cap, tile_chunks, 0);
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
  a.N = N; a.NB = NB; a.NC = NC; a.K = p->topk; a.SG = (int)SG; a.nS = (int)nS; a.B = p->block_size;
  a.status = d_status;

  layout_kernel<<<1, 1024, 0, st>>>(p->cu_seqlens, p->kv_doc_starts, N, p->total_tokens, p->kv_rows,
                                    p->block_size, NB, NC, blk_off, chunk_off, d_status);
  // shared memory: the staged piece, then per row of a window a counter
  // (pass 1) or a cursor (pass 4) and a chunk mask
  a.win = NB < kRowWindow ? NB : kRowWindow;
  const size_t count_smem = sizeof(K2QStage) + 2 * sizeof(int) * a.win;
  const size_t scatter_smem = sizeof(K2QStage) + 2 * sizeof(int) * a.win;
  if ((rc = cuda_status(cudaFuncSetAttribute(k2q_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)count_smem))) ||
      (rc = cuda_status(cudaFuncSetAttribute(k2q_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)scatter_smem))))
    return rc;
  k2q_count_kernel<<<dim3((unsigned)nS, Hi), kCountThreads, count_smem, st>>>(a);
  k2q_group_offsets_kernel<<<dim3((unsigned)((NB + 31) / 32), Hi), 1024, 0, st>>>(a);
  k2q_row_ptr_kernel<<<Hi, 1024, 0, st>>>(a);
  k2q_scatter_kernel<<<dim3((unsigned)nS, Hi), kScatterThreads, scatter_smem, st>>>(a);
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
  const int nh = key_tiles_per_block(p);
  const int64_t n = (int64_t)Hi * ntiles * NB * nh;
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
  a.edge_cap = edge_cap; a.task_cap = task_cap; a.N = N; a.NB = NB; a.NBt = NB * nh; a.NC = NC; a.Hi = Hi;
  a.tile_chunks = tile_chunks; a.ntiles = (int)ntiles; a.num_sms = num_sms; a.B = p->block_size; a.nh = nh;
  a.status = d_status;

  layout_kernel<<<1, 1024, 0, st>>>(p->cu_seqlens, p->kv_doc_starts, N, p->total_tokens, p->kv_rows,
                                    p->block_size, NB, NC, blk_off, chunk_off, d_status);
  if ((rc = cuda_status(cudaMemsetAsync(a.tcnt, 0, sizeof(int32_t) * n, st)))) return rc;
  const int64_t warps = (int64_t)Hi * NB * kRowParts;
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
  a.Hi = p->num_index_heads; a.nblk = (int)((items + kPlanBlock - 1) / kPlanBlock); a.B = p->block_size;
  a.status = d_status;
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
