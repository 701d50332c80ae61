// MSA block-sparse attention forward on sm_103a ("msa_bindings" page,
// sparse_atten_func, the flat forward): per (index head, query chunk) the 128
// rows (8 tokens x 16 q-heads) attend the chunk's selected key blocks
// causally, in one pass with an online softmax:
//   S_j = Q K_j^T (tcgen05, fp32 in TMEM), m = running row max (log2 units),
//   P_j = exp2(S_j - m) (bf16, in TMEM), l += rowsum(P_j),
//   O += P_j V_j (TMEM; the GEMM reads P_j from TMEM).
// The running max is moved only when a block raises it by more than kTau
// (so P stays below 2^kTau); O is then rescaled in TMEM by exp2(m_old - m_new).
// O = O / l is written as bf16 and LSE = (m + log2 l) ln 2, the form the
// backward consumes.
//
// Warps 0-3 run the softmax, one row per thread; warp 4 loads tiles (TMA) and
// issues the GEMMs.  They hand off through mbarriers: S_j full (MMA commit),
// S_j read (softmax), P_j written (softmax), P_j V_j done (MMA commit).  TMEM
// holds one S buffer, two P buffers and O: S_{j+1} is computed as soon as
// block j's softmax has read S_j, while P_j V_j runs from the other P buffer.
// K and V are double-buffered in smem and loaded ahead.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa_common.cuh"
#include "msa_host.cuh"
#include "msa_tmap.cuh"

namespace msa {

namespace fwd {
constexpr int kThreads = 160;       // 4 softmax warps + 1 load/MMA warp
constexpr int kIssueWarp = 4;
constexpr uint32_t OFF_Q = 0;       // [2 halves][128 rows][128 B]
constexpr uint32_t OFF_K = 32768;   // 2 buffers x [2 halves][64 keys][128 B]
constexpr uint32_t OFF_V = 65536;   // 2 buffers x [2 halves][64 keys][128 B]
constexpr uint32_t OFF_BAR = 98304;
constexpr uint32_t BAR_BYTES = 512;  // barriers, TMEM slot, the item's key-tile list
// Slack for aligning the dynamic window to 1024 B.  A window that would need
// more than this is reported.
constexpr uint32_t ALIGN_SLACK = 768;
constexpr uint32_t SMEM = OFF_BAR + BAR_BYTES + ALIGN_SLACK;
constexpr uint32_t TMEM_COLS = 256;
constexpr int kMaxTiles = 64;  // 64-key tiles of an item: up to 32 blocks of 128 keys
constexpr uint32_t COL_S = 0, COL_P = 64, COL_O = 128;  // S 64 columns, P 2 x 32 (bf16 pairs), O 128
constexpr float kTau = 8.f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace fwd

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 lanes x 32 bit, 32 consecutive columns per thread (thread t -> lane base+t).
__device__ __forceinline__ void tmem_st32x(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem], bf16 inputs, fp32 accumulate.  A is M rows
// on TMEM lanes, K-major, two bf16 per 32-bit column (lower k in the low half).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct FwdArgs {
  const int32_t* sel;
  const int32_t* plan;  // scheduler_metadata rows of a forward plan, or null: items in index order
  const int32_t* cu;
  const int32_t* chunk_off;
  uint16_t* o;
  float* lse;
  int N, NC, K, Hi, Hq;
  int nh;  // 64-key tiles per selected block (1 or 2)
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

// Both halves (64 of the 128 head dims each) of one 64-key K or V block.
__device__ __forceinline__ void load_kv(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int hi, int row) {
  mbar_arrive_expect_tx(bar, 16384u);
  tma_load_3d(dst, map, bar, 0, hi, row);
  tma_load_3d(dst + 8192, map, bar, 64, hi, row);
}

__global__ void __launch_bounds__(fwd::kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const int32_t* kv_doc_starts, FwdArgs a) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  const uintptr_t pad = ((raw + 1023) & ~uintptr_t(1023)) - raw;
  if (pad > ALIGN_SLACK) {  // uniform across the block: nothing has started yet
    if (threadIdx.x == 0) set_status(a.status, MSA_ERR_CUDA);
    return;
  }
  uint8_t* sm = smem_raw + pad;
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_pv = bar_q + 1;     // P V done (MMA commit)
  uint64_t* bar_k = bar_q + 2;      // two
  uint64_t* bar_v = bar_q + 4;      // two
  uint64_t* bar_s = bar_q + 6;      // S full (MMA commit)
  uint64_t* bar_sfree = bar_q + 7;  // S read (4 softmax warps)
  // two: P written and O rescaled (4 softmax warps), one per P buffer.
  // Block j+1's softmax signals only after P V of block j, which itself
  // follows the issuer's wait for block j, so one would do; two keep the
  // issuer's wait independent of that ordering.
  uint64_t* bar_pfull = bar_q + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_q + 11);
  // the item's 64-key tiles (up to 2 per selected block), count at [kMaxTiles]
  int* s_blocks = reinterpret_cast<int*>(bar_q + 12);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_pv, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_k[i], 1);
      mbar_init(&bar_v[i], 1);
      mbar_init(&bar_pfull[i], 4);
    }
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
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t sbase = smem_u32(sm);
  constexpr uint32_t ID_S = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t ID_O = idesc_bf16_f32(128, 128, false, true);
  // Blocks processed so far by this CTA: block n uses K/V/P buffer n & 1 and
  // phase parity (n >> 1) & 1 of their barriers, parity n & 1 of bar_s,
  // bar_sfree and bar_pv (one phase per block).
  uint32_t seq = 0, ph_q = 0;
  bool aborted = status_bad(a.status);
  const int64_t items = (int64_t)a.Hi * a.NC;
  for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
    // the walk's w-th item: the plan's row w (a permutation of the items,
    // longest first), or item w itself
    const int hi = a.plan ? a.plan[w * MSA_TASK_META_COLS] : (int)(w / a.NC);
    const int g = a.plan ? a.plan[w * MSA_TASK_META_COLS + 1] : (int)(w % a.NC);
    const int d = doc_of_chunk(a.chunk_off, a.N + 1, g);
    if (warp == kIssueWarp) {
      // compact the item's selection into 64-key tiles, order kept: a 128-key
      // block gives its lower tile and, when the chunk's last query reaches
      // it, its upper tile
      const int b = lane < a.K ? a.sel[((int64_t)hi * a.NC + g) * a.K + lane] : -1;
      int ntl = 0;
      if (b >= 0) {
        ntl = 1;
        if (a.nh > 1) {
          const int c = g - a.chunk_off[d];
          const int last = min(c * 8 + 7, a.cu[d + 1] - a.cu[d] - 1);
          ntl = (b * 128 + 64 <= last) ? 2 : 1;
        }
      }
      int x = ntl;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o2);
        if (lane >= o2) x += y;
      }
      const int at = x - ntl;
      for (int i = 0; i < ntl; ++i) s_blocks[at + i] = b * a.nh + i;
      if (lane == 31) s_blocks[fwd::kMaxTiles] = x;
    }
    if (__syncthreads_or(aborted)) break;
    const int nblk = s_blocks[fwd::kMaxTiles];
    const int kv0 = kv_doc_starts[d];
    const uint32_t seq0 = seq;
    if (warp == kIssueWarp) {
      // ---------------- loads and GEMMs ----------------
      // Every MMA of the previous item has completed: all buffers are free.
      if (nblk > 0) {
        const int c = g - a.chunk_off[d];
        const int tok0 = a.cu[d] + c * 8;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar_q, 32768u);
          tma_load_3d(sm + OFF_Q, &tmQ, bar_q, 0, hi * 16, tok0);
          tma_load_3d(sm + OFF_Q + 16384, &tmQ, bar_q, 64, hi * 16, tok0);
          for (int j = 0; j < 2 && j < nblk; ++j) {
            const uint32_t bf = (seq0 + j) & 1;
            load_kv(sm + OFF_K + bf * 16384, &tmK, &bar_k[bf], hi, kv0 + s_blocks[j] * 64);
            load_kv(sm + OFF_V + bf * 16384, &tmV, &bar_v[bf], hi, kv0 + s_blocks[j] * 64);
          }
        }
        __syncwarp();
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar_q, ph_q, a.status) &&
                                              mbar_wait(&bar_k[seq0 & 1], (seq0 >> 1) & 1, a.status));
        ph_q ^= 1;
        if (ok) {
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
              umma_bf16(tmem + COL_S, sdesc_sw128(sbase + OFF_Q + half * 16384 + sub, 16, 1024),
                        sdesc_sw128(sbase + OFF_K + (seq0 & 1) * 16384 + half * 8192 + sub, 16, 1024), ID_S,
                        kk > 0);
            }
            umma_commit(bar_s);
          }
          __syncwarp();
        }
        for (int j = 0; j < nblk && ok; ++j) {
          const uint32_t n = seq0 + j, bf = n & 1;
          // S_{j+1} once K_{j+1} has landed and every softmax warp has read S_j;
          // then K_{j+2} into the K buffer S_j read (S_j completed before it was read)
          if (j + 1 < nblk) {
            const uint32_t n1 = n + 1, b1 = n1 & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_k[b1], (n1 >> 1) & 1, a.status) &&
                                             mbar_wait(bar_sfree, n & 1, a.status));
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
                umma_bf16(tmem + COL_S, sdesc_sw128(sbase + OFF_Q + half * 16384 + sub, 16, 1024),
                          sdesc_sw128(sbase + OFF_K + b1 * 16384 + half * 8192 + sub, 16, 1024), ID_S, kk > 0);
              }
              umma_commit(bar_s);
              if (j + 2 < nblk) load_kv(sm + OFF_K + bf * 16384, &tmK, &bar_k[bf], hi, kv0 + s_blocks[j + 2] * 64);
            }
            __syncwarp();
          }
          // V_{j+1} into the V buffer P V of block j-1 read, once that has completed
          if (j >= 1 && j + 1 < nblk) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_pv, (n - 1) & 1, a.status)))) break;
            if (elect_one())
              load_kv(sm + OFF_V + (bf ^ 1) * 16384, &tmV, &bar_v[bf ^ 1], hi, kv0 + s_blocks[j + 1] * 64);
            __syncwarp();
          }
          // O += P_j V_j once P_j is written and V_j has landed
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bar_pfull[bf], (n >> 1) & 1, a.status) &&
                              mbar_wait(&bar_v[bf], (n >> 1) & 1, a.status));
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ts(tmem + COL_O, tmem + COL_P + bf * 32 + kk * 8,
                           sdesc_sw128(sbase + OFF_V + bf * 16384 + kk * 2048, 8192, 1024), ID_O,
                           (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit(bar_pv);
          }
          __syncwarp();
        }
        if (!ok) aborted = true;
      }
    } else {
      // ---------------- softmax, one row per thread ----------------
      const int c = g - a.chunk_off[d];
      const int len = a.cu[d + 1] - a.cu[d];
      const int tok0 = a.cu[d] + c * 8;
      const int qcount = min(8, len - c * 8);
      const int slot = tid >> 4, hh = tid & 15;
      const int qpos = slot < qcount ? c * 8 + slot : -1;
      float m_run = -CUDART_INF_F, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < nblk; ++j) {
        const uint32_t n = seq0 + j, bf = n & 1;
        const int b = s_blocks[j];
        ok = __all_sync(0xffffffffu, mbar_wait(bar_s, n & 1, a.status));
        if (!ok) break;
        tc_fence_after();
        // raw scores; keys after the row's query masked to -inf.  A block that
        // ends before the chunk's first query needs no mask: every key precedes
        // every real row, and rows past the document end (their queries are
        // real tokens or TMA zero fill, so finite) are never stored.
        const bool full = b * 64 + 63 <= c * 8;
        float xs[64];
        {
          uint32_t sv0[32], sv1[32];
          tmem_ld32x(tmem + lane_base + COL_S, sv0);
          tmem_ld32x(tmem + lane_base + COL_S + 32, sv1);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            xs[e] = __uint_as_float(sv0[e]);
            xs[32 + e] = __uint_as_float(sv1[e]);
          }
        }
        if (!full) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (b * 64 + e > qpos) xs[e] = -CUDART_INF_F;
        }
        float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int e = 0; e < 64; e += 8) {
#pragma unroll
          for (int r = 0; r < 4; ++r) m4[r] = max3(m4[r], xs[e + 2 * r], xs[e + 2 * r + 1]);
        }
        const float smax = max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        // S_j is in registers: the next S GEMM may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree);
        const float bmax = smax * a.scale_log2;  // log2 units (scale > 0)
        const bool upd = bmax > m_run + kTau;    // also true for the row's first key
        const bool resc = upd && m_run > -CUDART_INF_F;
        const float alpha = upd ? ex2_approx(m_run - bmax) : 1.f;
        if (upd) {
          l_run *= alpha;
          m_run = bmax;
        }
        // p = exp2(x scale - m); masked keys give exp2(-inf) = 0, and a row
        // with no key yet (m = -inf) uses 0 for m so nothing is inf - inf
        const float nm = m_run > -CUDART_INF_F ? -m_run : 0.f;
        uint32_t pk[32];
        const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nm2 = f2_pack(nm, nm);
        uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          float y0, y1;
          f2_unpack(f2_fma(f2_pack(xs[e], xs[e + 1]), sc2, nm2), y0, y1);
          const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
          ls2[(e >> 1) & 1] = f2_add(ls2[(e >> 1) & 1], f2_pack(p0, p1));
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(ls2[0], a0, a1);
          f2_unpack(ls2[1], b0, b1);
          l_run += (a0 + a1) + (b0 + b1);
        }
        if (__any_sync(0xffffffffu, resc)) {  // warp-collective TMEM access
          // P V of block j-1 has accumulated into O (j > 0: no row has O yet at j = 0)
          ok = __all_sync(0xffffffffu, mbar_wait(bar_pv, (n - 1) & 1, a.status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32x(tmem + lane_base + COL_O + c0, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32x(tmem + lane_base + COL_O + c0, ov);
          }
          tmem_st_wait();
        }
        // P_j into P buffer bf, which P V of block j-2 read: this warp waited
        // for that P V in block j-1, before it signalled P_{j-1}
        tmem_st32x(tmem + lane_base + COL_P + bf * 32, pk);
        tmem_st_wait();
        // Consume P V of block j-1 before signalling P_j, so this warp takes
        // bar_pv's phases in order: P V of block j-2 was consumed in block j-1
        // and P V of block j cannot start before the signal.
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar_pv, (n - 1) & 1, a.status));
          if (!ok) break;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pfull[bf]);
      }
      if (ok && nblk > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar_pv, (seq0 + nblk - 1) & 1, a.status));
      if (!ok) {
        aborted = true;
      } else {
        tc_fence_after();
        // epilogue: O / l -> bf16 global, LSE natural log.  TMEM loads are
        // warp-collective, so every thread loads and only real rows store.
        const int64_t row = (int64_t)(tok0 + slot) * a.Hq + hi * 16 + hh;
        if (qpos >= 0) a.lse[row] = l_run > 0.f ? (m_run + lg2_approx(l_run)) * kLn2 : -CUDART_INF_F;
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(a.o + row * 128);
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[32];
          if (nblk > 0) {
            tmem_ld32x(tmem + lane_base + COL_O + c0, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          if (qpos >= 0) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[c0 / 8 + q4] = make_uint4(
                  pack_bf16x2(__uint_as_float(v[8 * q4 + 0]) * inv, __uint_as_float(v[8 * q4 + 1]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * q4 + 2]) * inv, __uint_as_float(v[8 * q4 + 3]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * q4 + 4]) * inv, __uint_as_float(v[8 * q4 + 5]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * q4 + 6]) * inv, __uint_as_float(v[8 * q4 + 7]) * inv));
          }
        }
      }
    }
    seq = seq0 + nblk;
    // all of the item's MMAs have completed and its O has been read
    tc_fence_before();
    if (__syncthreads_or(aborted)) break;
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// defined in msa_tables.cu
__global__ void layout_kernel(const int32_t* cu, const int32_t* kvs, int N, int T, int W, int B, int NB, int NC,
                              int32_t* blk_off, int32_t* chunk_off, int32_t* status);

}  // namespace msa

using namespace msa;

static int launch_fwd(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const int32_t* sel, const int32_t* plan, uint16_t* o, float* lse, int32_t* d_status, void* ws,
                      size_t ws_bytes, void* stream) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (plan && !aligned16(plan)) return MSA_ERR_INVALID_ARGUMENT;
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
                                    p->block_size, p->num_blocks, p->num_chunks, blk_off, chunk_off, d_status);
  // The largest shared-memory carveout: two CTAs of ~97 KB share one SM.
  if (cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fwd::SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return MSA_ERR_CUDA;
  FwdArgs a;
  a.sel = sel; a.plan = plan; a.cu = p->cu_seqlens; a.chunk_off = chunk_off; a.o = o; a.lse = lse; a.N = N;
  a.NC = p->num_chunks; a.K = p->topk; a.Hi = p->num_index_heads; a.Hq = (int)Hq; a.nh = key_tiles_per_block(p);
  a.scale_log2 = p->softmax_scale * fwd::kLog2e; a.status = d_status;
  const int64_t items = (int64_t)p->num_index_heads * p->num_chunks;
  // CTAs resident per SM: shared memory per SM over this CTA's share (with
  // the per-block reservation), at most two (two 256-column TMEM allocations).
  int dev = 0, smem_sm = 0, smem_rsv = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
    return MSA_ERR_CUDA;
  int per_sm = smem_sm / ((int)fwd::SMEM + smem_rsv);
  if (per_sm > 2) per_sm = 2;
  if (per_sm < 1) return MSA_ERR_CUDA;
  const int64_t slots = (int64_t)per_sm * sms;
  const int grid = (int)(items < slots ? items : slots);
  fwd_kernel<<<grid, fwd::kThreads, fwd::SMEM, st>>>(tmQ, tmK, tmV, p->kv_doc_starts, a);
  return cuda_status(cudaGetLastError());
}

extern "C" int msa_fwd(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* sel, uint16_t* o, float* lse, int32_t* d_status, void* ws, size_t ws_bytes,
                       void* stream) {
  return launch_fwd(p, q, k, v, sel, nullptr, o, lse, d_status, ws, ws_bytes, stream);
}

extern "C" int msa_fwd_planned(const msa_problem* p, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* sel, const int32_t* scheduler_metadata, uint16_t* o, float* lse,
                               int32_t* d_status, void* ws, size_t ws_bytes, void* stream) {
  if (!scheduler_metadata) return MSA_ERR_INVALID_ARGUMENT;
  return launch_fwd(p, q, k, v, sel, scheduler_metadata, o, lse, d_status, ws, ws_bytes, stream);
}
