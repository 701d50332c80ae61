// Warp-specialised, pipelined main backward kernel (sm_103a).
//
// Roles (24 warps, 768 threads, one CTA per SM, persistent over the walk):
//   warp 0      task-info producer: walks the CTA's task sequence up to
//               kInfo tasks ahead and publishes, per task, its index head,
//               key block, K/V row, token row, query positions and bucket
//               segment flags in a shared-memory ring, so no other role reads
//               task tables from global memory on its critical path.
//   warp 1      TMA producer: K/V once per bucket segment, Q/dO per task into
//               a 2-stage ring.
//   warp 2      MMA issuer A: S = Q K^T as soon as Q has landed, then
//               dP = dO V^T once dO has.
//   warp 3      MMA issuer B: dK^T += Q^T dS, dV^T += dO^T P and
//               dQ = dS K.  Two issuing threads keep the tensor core fed while
//               each waits on its own dependencies; their TMEM targets are
//               disjoint and every cross-phase ordering goes through an
//               mbarrier.
//   warps 4-19  softmax / dS: TMEM -> registers -> P, dS (bf16, swizzled
//               shared memory).  Warp w owns TMEM lanes 32*(w%4).. and key
//               columns 16*((w-4)/4)..; four per SM sub-partition, so the
//               latency of one warp's exp/convert chain hides behind others'.
//   warps 20-23 reduce: dQ per task and dK/dV per segment, TMEM -> swizzled
//               staging (bf16 dQ, or fp32 with the fp32 dQ option; fp32 dK/dV;
//               two 4 KB slots per warp, so a slot is refilled while the
//               reduce-add of the other is still reading) -> TMA bulk
//               reduce-add.
//
// Issuer A issues S, then dP (each its own accumulator chain, so S can start
// before the dO tile lands); issuer B issues the dK^T chain, then the dV^T
// chain, then dQ, and waits for every buffer it needs before it waits for
// P/dS, so that nothing but the hand-off itself separates P/dS landing from
// the first MMA.
//
// A task's Q tile is held from its TMA load until its dK^T MMAs have run and
// its dO tile until its dV^T MMAs have (dQ reads only dS and K), so the load
// of the task two ahead into the Q half starts one chain before the dO half,
// and both start before the dQ MMAs.  dQ is double-buffered in TMEM, so the
// dQ MMAs of task j+1 never wait for the drain of task j.
//
// TMEM (512 columns): S at 0, dP at 64, dQ[2] at 128/256 (128 cols each),
// dK^T at 384, dV^T at 448 (64 cols each; lane = head-dim index).
//
// Every mbarrier wait is bounded (kWaitLimitNs) and also gives up when any
// role has raised the shared abort flag; the status word records the timeout.
// On the way out the TMA producer waits (bounded, ignoring the abort flag) for
// every load it issued, so no copy still writes shared memory when the CTA
// exits; the issuers wait for their last MMAs before TMEM is freed.
#pragma once

namespace msa {
namespace ws {

constexpr int kWarps = 24;
constexpr int kThreads = kWarps * 32;
constexpr int kInfoWarp = 0, kLoadWarp = 1, kMmaWarp = 2, kMmaBWarp = 3, kComp0 = 4, kNumComp = 16, kRed0 = 20,
              kNumRed = 4;
constexpr int kInfo = 8;  // task-info ring entries

constexpr uint32_t OFF_QDO = 0;          // 2 stages x (Q 32 KB | dO 32 KB)
constexpr uint32_t QDO_STAGE = 65536;
constexpr uint32_t DO_IN_STAGE = 32768;
constexpr uint32_t OFF_K = 131072;       // 16 KB, [64 keys][128 dims] bf16 (two 64-dim halves)
constexpr uint32_t OFF_V = 147456;       // 16 KB
constexpr uint32_t OFF_P = 163840;       // 16 KB, [128 rows][64 keys] bf16
constexpr uint32_t OFF_DS = 180224;      // 16 KB
constexpr uint32_t OFF_ST = 196608;      // 4 warps x 2 slots x 4 KB fp32 staging
constexpr uint32_t OFF_BAR = 229376;    // barriers, then the task-info ring
constexpr uint32_t SMEM = OFF_BAR + 1024 + 1024;

enum : int {
  Q_FULL = 0, Q_EMPTY = 2, DO_FULL = 4, DO_EMPTY = 6, KV_FULL = 8, K_EMPTY = 9, V_EMPTY = 10, S_FULL = 11,
  S_EMPTY = 12, PDS_FULL = 13, PDS_EMPTY = 14, DQ_FULL = 15, DQ_EMPTY = 17, DKV_FULL = 19, DKV_EMPTY = 20,
  DRAIN = 21, INFO_FULL = 22, INFO_EMPTY = INFO_FULL + kInfo, NUM_BARS = INFO_EMPTY + kInfo
};

// One task as every role needs it.
struct TaskInfo {
  int32_t hi, tok0, b, kvrow;
  int32_t flags;          // bit 0: first task of its bucket segment, bit 1: last
  uint32_t seg;           // segment ordinal within this CTA's sequence
  int32_t pad[2];
  int32_t qpos[8];        // document-local position of each token slot, -1 = empty
};
static_assert(sizeof(TaskInfo) == 64, "task info entry");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_DP = 64, COL_DK = 384, COL_DV = 448;
__device__ __forceinline__ uint32_t col_dq(uint32_t buf) { return 128 + buf * 128; }

// The CTA's task sequence.  The walk's units are the pages' (full units of R
// consecutive rows, then tail units of rows strided by the tail-unit count),
// but a CTA takes its next unit from a global counter when it has finished the
// last one, instead of the static unit blockIdx.x + k * gridDim.x: the CTAs
// then stay within a few units of one another in the row order, which keeps
// the query tiles they touch at the same time small enough to stay in L2.
struct Walk {
  int n, R, full, grid;
  int u, i, cnt, t0, step;
  int32_t* ctr;
  __device__ __forceinline__ void setup() {
    if (u >= grid) return;
    if (u < full) {
      t0 = u * R; step = 1; cnt = R;
    } else {
      step = grid - full; t0 = full * R + (u - full); cnt = (n - t0 + step - 1) / step;
    }
  }
  __device__ __forceinline__ void init(const int32_t* walk, int32_t* unit_ctr) {
    n = walk[MSA_WALK_ROWS]; R = walk[MSA_WALK_ROWS_PER_CTA];
    full = walk[MSA_WALK_FULL]; grid = walk[MSA_WALK_GRID];
    ctr = unit_ctr;
    u = atomicAdd(ctr, 1); i = 0;
    setup();
  }
  __device__ __forceinline__ int take() {  // current task or -1, then advance
    if (u >= grid) return -1;
    const int t = t0 + i * step;
    if (++i >= cnt) { u = atomicAdd(ctr, 1); i = 0; setup(); }
    return t;
  }
};

// Current / next task of the sequence, with the bucket key of each.
struct Seq {
  Walk w;
  int cur, nxt;
  __device__ __forceinline__ void init(const int32_t* walk, int32_t* unit_ctr) {
    w.init(walk, unit_ctr);
    cur = w.take();
    nxt = w.take();
  }
  __device__ __forceinline__ void advance() {
    cur = nxt;
    nxt = w.take();
  }
};

__device__ __forceinline__ int64_t bucket_key(const int32_t* meta, int t) {
  return (static_cast<int64_t>(meta[(int64_t)t * MSA_TASK_META_COLS]) << 32) |
         static_cast<uint32_t>(meta[(int64_t)t * MSA_TASK_META_COLS + 1]);
}

struct Shared {
  uint64_t bar[NUM_BARS];
  uint32_t tmem_base;
  int abort;
  int32_t pad[6];
  TaskInfo info[kInfo];
};
static_assert(sizeof(Shared) <= 1024, "shared control block");

// Single-thread wait.  Gives up (false) on timeout, or as soon as another role
// has aborted unless honor_abort is false (used for the final MMA drain).
__device__ __forceinline__ bool wait_bar(Shared* sh, int idx, uint32_t parity, int32_t* status,
                                         bool honor_abort = true) {
  uint64_t* bar = &sh->bar[idx];
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *reinterpret_cast<volatile int*>(&sh->abort)) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      set_status(status, MSA_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sh->abort) = 1;
      return false;
    }
  }
}

// Warp-level wait: lane 0 polls, the outcome is broadcast so the warp stays
// converged for the warp-collective tcgen05.ld that follows.
__device__ __forceinline__ bool wait_bar_warp(Shared* sh, int idx, uint32_t parity, int32_t* status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(sh, idx, parity, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// 32 consecutive TMEM columns of this warp's lane quarter into registers.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&v)[32]) {
  tmem_ld16(addr, *reinterpret_cast<uint32_t(*)[16]>(v));
  tmem_ld16(addr + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
  tmem_ld_wait();
}

// 16 keys of row m (8 packed bf16 pairs) into the 128B-swizzled
// [128 rows][64 keys] bf16 tile at base; qtr selects keys 16*qtr .. 16*qtr+15.
__device__ __forceinline__ void store_row16(uint8_t* base, int m, int qtr, const uint32_t (&pk)[8]) {
  uint8_t* row = base + m * 128;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t o = static_cast<uint32_t>(((qtr * 2 + c) ^ (m & 7)) << 4);
    *reinterpret_cast<uint4*>(row + o) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  }
}

}  // namespace ws

// kDqFp32: dQ tiles are reduce-added in fp32 into the workspace accumulator
// (tmdQ maps it) instead of in bf16 into the output; two instances, so the
// default path carries no branch for the option.  kHoldReduce (a self-test of
// the bounded waits, never a result): the reduce warps stay idle, so the
// hand-offs that wait for them run out their limit and every role aborts.
template <bool kDqFp32, bool kHoldReduce = false>
__global__ void __launch_bounds__(ws::kThreads, 1)
    bwd_main_ws(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
                const __grid_constant__ CUtensorMap tmdV, MainArgs a) {
  using namespace ws;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared* sh = reinterpret_cast<Shared*>(sm + OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // TMA-filled and MMA-committed barriers take one arrival; the softmax
    // warps' hand-offs (S/dP drained, P/dS stored) take one per softmax warp;
    // the reduce warps' (dQ, dK/dV drained) one per reduce warp; DRAIN one
    // per issuer.
    uint32_t counts[INFO_FULL];
    for (int i = 0; i < INFO_FULL; ++i) counts[i] = 1;
    counts[S_EMPTY] = counts[PDS_FULL] = kNumComp;
    counts[DQ_EMPTY] = counts[DQ_EMPTY + 1] = counts[DKV_EMPTY] = kNumRed;
    counts[DRAIN] = 2;
    for (int i = 0; i < INFO_FULL; ++i) mbar_init(&sh->bar[i], counts[i]);
    for (int i = 0; i < kInfo; ++i) {
      mbar_init(&sh->bar[INFO_FULL + i], 1);
      mbar_init(&sh->bar[INFO_EMPTY + i], kNumRed);
    }
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sh->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const int32_t* meta = a.meta;

  if (!status_bad(a.status)) {
    if (warp == kInfoWarp) {
      // ------------------------------------------------------------ task info
      if (lane == 0) {
        Seq s;
        s.init(a.walk, a.unit_ctr);
        uint32_t j = 0, nseg = 0;
        int64_t prev = -1;
        int64_t key = s.cur >= 0 ? bucket_key(meta, s.cur) : -1;
        while (s.cur >= 0) {
          const int t = s.cur;
          const int64_t nkey = s.nxt >= 0 ? bucket_key(meta, s.nxt) : -2;
          const int32_t* mt = meta + (int64_t)t * MSA_TASK_META_COLS;
          const int hi = mt[0], d = mt[4], b = mt[5];
          const int tok0 = a.q_rows[(int64_t)t * 8];
          const int4 qp0 = *reinterpret_cast<const int4*>(a.q_pos + (int64_t)t * 8);
          const int4 qp1 = *reinterpret_cast<const int4*>(a.q_pos + (int64_t)t * 8 + 4);
          const int kvrow = a.kv_doc_starts[d] + b * 64;
          const bool first = key != prev;
          if (first) ++nseg;
          const uint32_t slot = j % kInfo;
          if (!wait_bar(sh, INFO_EMPTY + slot, ((j / kInfo) & 1) ^ 1, a.status)) break;
          TaskInfo& e = sh->info[slot];
          e.hi = hi; e.tok0 = tok0; e.b = b; e.kvrow = kvrow;
          e.flags = (first ? 1 : 0) | (nkey != key ? 2 : 0);
          e.seg = nseg - 1;
          e.qpos[0] = qp0.x; e.qpos[1] = qp0.y; e.qpos[2] = qp0.z; e.qpos[3] = qp0.w;
          e.qpos[4] = qp1.x; e.qpos[5] = qp1.y; e.qpos[6] = qp1.z; e.qpos[7] = qp1.w;
          mbar_arrive(&sh->bar[INFO_FULL + slot]);
          prev = key;
          key = nkey;
          ++j;
          s.advance();
        }
        // a sentinel entry tells every consumer that the sequence has ended
        const uint32_t slot = j % kInfo;
        if (wait_bar(sh, INFO_EMPTY + slot, ((j / kInfo) & 1) ^ 1, a.status)) {
          sh->info[slot].hi = -1;
          mbar_arrive(&sh->bar[INFO_FULL + slot]);
        }
      }
    } else if (warp == kLoadWarp) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        // Q/dO tiles are reused by every task of their query chunk within the
        // query tile (they stay in L2 while the CTAs walk the tile together);
        // a K/V tile only within its bucket segment
        const uint64_t keep = l2_evict_last(), stream = l2_evict_first();
        // parity of the last phase armed on each FULL barrier (-1: none), so
        // that loads still in flight can be waited for on the way out
        int armed_q[2] = {-1, -1}, armed_do[2] = {-1, -1}, armed_kv = -1;
        for (uint32_t j = 0;; ++j) {
          const uint32_t slot = j % kInfo;
          if (!wait_bar(sh, INFO_FULL + slot, (j / kInfo) & 1, a.status)) break;
          const TaskInfo& e = sh->info[slot];
          const int hi = e.hi;
          if (hi < 0) break;
          if (e.flags & 1) {
            const uint32_t seg = e.seg;
            if (!wait_bar(sh, K_EMPTY, (seg & 1) ^ 1, a.status)) break;
            if (!wait_bar(sh, V_EMPTY, (seg & 1) ^ 1, a.status)) break;
            uint64_t* fb = &sh->bar[KV_FULL];
            mbar_arrive_expect_tx(fb, 32768u);
            tma_load_3d_hint(sm + OFF_K, &tmK, fb, 0, hi, e.kvrow, stream);
            tma_load_3d_hint(sm + OFF_K + 8192, &tmK, fb, 64, hi, e.kvrow, stream);
            tma_load_3d_hint(sm + OFF_V, &tmV, fb, 0, hi, e.kvrow, stream);
            tma_load_3d_hint(sm + OFF_V + 8192, &tmV, fb, 64, hi, e.kvrow, stream);
            armed_kv = (int)(seg & 1);
          }
          const uint32_t qst = j & 1, qph = ((j >> 1) & 1) ^ 1;
          uint8_t* st = sm + OFF_QDO + qst * QDO_STAGE;
          if (!wait_bar(sh, Q_EMPTY + qst, qph, a.status)) break;
          mbar_arrive_expect_tx(&sh->bar[Q_FULL + qst], 32768u);
          tma_load_3d_hint(st, &tmQ, &sh->bar[Q_FULL + qst], 0, hi * 16, e.tok0, keep);
          tma_load_3d_hint(st + 16384, &tmQ, &sh->bar[Q_FULL + qst], 64, hi * 16, e.tok0, keep);
          armed_q[qst] = (int)(qph ^ 1);
          if (!wait_bar(sh, DO_EMPTY + qst, qph, a.status)) break;
          mbar_arrive_expect_tx(&sh->bar[DO_FULL + qst], 32768u);
          tma_load_3d_hint(st + DO_IN_STAGE, &tmdO, &sh->bar[DO_FULL + qst], 0, hi * 16, e.tok0, keep);
          tma_load_3d_hint(st + DO_IN_STAGE + 16384, &tmdO, &sh->bar[DO_FULL + qst], 64, hi * 16, e.tok0, keep);
          armed_do[qst] = (int)(qph ^ 1);
        }
        // Every load issued has landed before the CTA can exit: after an abort
        // some were never consumed.  One phase at most is pending per barrier
        // (a barrier is re-armed only after its last phase was consumed), and
        // on a normal exit each of these waits returns at once.
        for (int s2 = 0; s2 < 2; ++s2) {
          if (armed_q[s2] >= 0) wait_bar(sh, Q_FULL + s2, (uint32_t)armed_q[s2], a.status, false);
          if (armed_do[s2] >= 0) wait_bar(sh, DO_FULL + s2, (uint32_t)armed_do[s2], a.status, false);
        }
        if (armed_kv >= 0) wait_bar(sh, KV_FULL, (uint32_t)armed_kv, a.status, false);
      }
    } else if (warp == kMmaWarp || warp == kMmaBWarp) {
      // ------------------------------------------------------------ MMA issuers
      // The whole warp runs the loop, so waits, task info and descriptors are
      // warp-uniform; one elected lane issues each burst of MMAs and its
      // commits.  (Issuing from a lone lane costs about 1.6x more per MMA.)
      constexpr uint32_t ID_S = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t ID_T = idesc_bf16_f32(128, 64, true, true);
      constexpr uint32_t ID_Q = idesc_bf16_f32(128, 128, false, true);
      const uint32_t sb = smem_u32(sm);
      // Descriptor bases; a K step or a stage is an immediate added to the
      // 14-bit start-address field (byte offset >> 4; all addresses < 256 KB).
      constexpr uint64_t kStageQ = QDO_STAGE >> 4;
      const bool is_a = warp == kMmaWarp;
      for (uint32_t j = 0;; ++j) {
        const uint32_t slot = j % kInfo;
        if (!wait_bar_warp(sh, INFO_FULL + slot, (j / kInfo) & 1, a.status)) break;
        const TaskInfo& e = sh->info[slot];
        const int hi = e.hi, flags = e.flags;
        const uint32_t seg = e.seg;
        __syncwarp();
        if (hi < 0) break;
        const bool first = flags & 1, last = (flags >> 1) & 1;
        const uint32_t st = j & 1, ph = (j >> 1) & 1;  // Q/dO stage and dQ buffer
        if (is_a) {
          // S = Q K^T, then dP = dO V^T
          if (first && !wait_bar_warp(sh, KV_FULL, seg & 1, a.status)) break;
          if (!wait_bar_warp(sh, S_EMPTY, (j & 1) ^ 1, a.status)) break;
          const uint64_t qk = sdesc_sw128(sb + OFF_QDO, 16, 1024) + st * kStageQ;
          const uint64_t kk0 = sdesc_sw128(sb + OFF_K, 16, 1024);
          const uint64_t dok = sdesc_sw128(sb + OFF_QDO + DO_IN_STAGE, 16, 1024) + st * kStageQ;
          const uint64_t vk = sdesc_sw128(sb + OFF_V, 16, 1024);
          // S as soon as Q has landed, dP once dO has
          if (!wait_bar_warp(sh, Q_FULL + st, ph, a.status)) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ao = (kk >> 2) * 1024 + (kk & 3) * 2, bo = (kk >> 2) * 512 + (kk & 3) * 2;
              umma_bf16(tmem + COL_S, qk + ao, kk0 + bo, ID_S, kk > 0);
            }
          }
          __syncwarp();
          if (!wait_bar_warp(sh, DO_FULL + st, ph, a.status)) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ao = (kk >> 2) * 1024 + (kk & 3) * 2, bo = (kk >> 2) * 512 + (kk & 3) * 2;
              umma_bf16(tmem + COL_DP, dok + ao, vk + bo, ID_S, kk > 0);
            }
            umma_commit(&sh->bar[S_FULL]);
            if (last) umma_commit(&sh->bar[V_EMPTY]);
          }
          __syncwarp();
        } else {
          // dK^T += Q^T dS, then dV^T += dO^T P, then dQ = dS K.  P/dS are
          // stored after S/dP completed, so once dK has run no MMA of the task
          // reads its Q tile and once dV has run none reads its dO tile: each
          // half of the stage is released as soon as its chain is done (a
          // single warp-issued chain runs as fast as two interleaved ones).
          if (first && !wait_bar_warp(sh, DKV_EMPTY, (seg & 1) ^ 1, a.status)) break;
          if (!wait_bar_warp(sh, DQ_EMPTY + st, ph ^ 1, a.status)) break;
          if (!wait_bar_warp(sh, PDS_FULL, j & 1, a.status)) break;
          tc_fence_after();
          const uint32_t acc0 = first ? 0u : 1u;
          const uint64_t dom = sdesc_sw128(sb + OFF_QDO + DO_IN_STAGE, 16384, 1024) + st * kStageQ;
          const uint64_t pm = sdesc_sw128(sb + OFF_P, 8192, 1024);
          const uint64_t qm = sdesc_sw128(sb + OFF_QDO, 16384, 1024) + st * kStageQ;
          const uint64_t dsm = sdesc_sw128(sb + OFF_DS, 8192, 1024);
          const uint64_t dsk = sdesc_sw128(sb + OFF_DS, 16, 1024);
          const uint64_t km = sdesc_sw128(sb + OFF_K, 8192, 1024);
          const uint32_t dq = tmem + col_dq(st);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16(tmem + COL_DK, qm + kk * 128, dsm + kk * 128, ID_T, kk > 0 ? 1u : acc0);
            umma_commit(&sh->bar[Q_EMPTY + st]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16(tmem + COL_DV, dom + kk * 128, pm + kk * 128, ID_T, kk > 0 ? 1u : acc0);
            umma_commit(&sh->bar[DO_EMPTY + st]);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) umma_bf16(dq, dsk + k4 * 2, km + k4 * 128, ID_Q, k4 > 0);
            umma_commit(&sh->bar[PDS_EMPTY]);
            umma_commit(&sh->bar[DQ_FULL + st]);
            if (last) {
              umma_commit(&sh->bar[K_EMPTY]);
              umma_commit(&sh->bar[DKV_FULL]);
            }
          }
          __syncwarp();
        }
      }
    } else if (warp < kRed0) {
      // ------------------------------------------------------------ softmax / dS
      const int sp = warp & 3, qtr = (warp - kComp0) >> 2;
      const int m = sp * 32 + lane, slot_row = m >> 4, hh = m & 15;
      const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
      // Per-row LSE and D of the next task, loaded one task ahead.  The raw
      // values are only consumed in the next iteration, so the loads stay in
      // flight across this task instead of stalling the warp here.
      auto fetch = [&](const TaskInfo& e, int& qpos, float& lse_raw, float& dlt_raw) {
        qpos = e.qpos[slot_row];
        const int64_t row = (int64_t)(e.tok0 + slot_row) * a.Hq + e.hi * 16 + hh;
        lse_raw = qpos >= 0 ? a.lse[row] : 0.f;
        dlt_raw = qpos >= 0 ? a.delta[row] : 0.f;
      };
      if (!wait_bar_warp(sh, INFO_FULL + 0, 0, a.status)) goto comp_done;
      {
        int qpos, nqpos = -1;
        float lse_raw, dlt_raw, nlse_raw = 0.f, ndlt_raw = 0.f;
        int b = sh->info[0].b;
        bool more = sh->info[0].hi >= 0;
        if (more) fetch(sh->info[0], qpos, lse_raw, dlt_raw);
        for (uint32_t j = 0; more; ++j) {
          // look ahead: next task's info and its per-row scalars
          const uint32_t nslot = (j + 1) % kInfo;
          if (!wait_bar_warp(sh, INFO_FULL + nslot, ((j + 1) / kInfo) & 1, a.status)) break;
          const TaskInfo& ne = sh->info[nslot];
          const bool nmore = ne.hi >= 0;
          const int nb = ne.b;
          if (nmore) fetch(ne, nqpos, nlse_raw, ndlt_raw);
          const uint32_t par = j & 1;
          const int kbase = b * 64 + qtr * 16;
          if (!wait_bar_warp(sh, S_FULL, par, a.status)) break;
          tc_fence_after();
          uint32_t sv[16], dpv[16];
          tmem_ld16(tmem + lane_base + COL_S + qtr * 16, sv);
          tmem_ld16(tmem + lane_base + COL_DP + qtr * 16, dpv);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->bar[S_EMPTY]);
          const float lse2 = lse_raw * kLog2e, dsc = dlt_raw * a.scale;
          // P = exp2(S * scale * log2e - LSE * log2e) on the causal mask and
          // dS = P * (dP * scale - D * scale); masked entries are exactly 0
          uint32_t pk[8], dk[8];
          const int lim = qpos - kbase;  // keys kbase + e with e <= lim are attended
          if (lim >= 15) {
            // the whole 16-key slice is attended (every block but the diagonal one)
            // paired fp32 FMA/multiply: each lane rounds as the scalar form would
            const uint64_t sl2 = f2_pack(a.scale_log2, a.scale_log2), nl2 = f2_pack(-lse2, -lse2);
            const uint64_t sc2 = f2_pack(a.scale, a.scale), nd2 = f2_pack(-dsc, -dsc);
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float y0, y1, d0, d1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2, nl2), y0, y1);
              const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
              const uint64_t t = f2_fma(f2_pack(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])), sc2, nd2);
              f2_unpack(f2_mul(f2_pack(p0, p1), t), d0, d1);
              pk[e >> 1] = pack_bf16x2(p0, p1);
              dk[e >> 1] = pack_bf16x2(d0, d1);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float p[2], ds[2];
#pragma unroll
              for (int x = 0; x < 2; ++x) {
                const bool valid = e + x <= lim;
                const float pv = ex2_approx(fmaf(__uint_as_float(sv[e + x]), a.scale_log2, -lse2));
                p[x] = valid ? pv : 0.f;
                ds[x] = valid ? pv * fmaf(__uint_as_float(dpv[e + x]), a.scale, -dsc) : 0.f;
              }
              pk[e >> 1] = pack_bf16x2(p[0], p[1]);
              dk[e >> 1] = pack_bf16x2(ds[0], ds[1]);
            }
          }
          if (!wait_bar_warp(sh, PDS_EMPTY, par ^ 1, a.status)) break;
          store_row16(sm + OFF_P, m, qtr, pk);
          store_row16(sm + OFF_DS, m, qtr, dk);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->bar[PDS_FULL]);
          qpos = nqpos; lse_raw = nlse_raw; dlt_raw = ndlt_raw; b = nb; more = nmore;
        }
      }
    comp_done:;
    } else {
      // ------------------------------------------------------------ reduce
      // Warp sp owns TMEM lanes 32*sp..: dQ rows of tokens 2*sp, 2*sp+1 and
      // head-dim rows 32*sp.. of dK^T/dV^T.  Each 4 KB chunk goes through one
      // of the warp's two staging slots as its own bulk group, so refilling a
      // slot only waits for the reduce-add issued two chunks earlier.
      const int sp = warp & 3;
      const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
      uint8_t* stg0 = sm + OFF_ST + (warp - kRed0) * 8192;
      uint32_t chunk = 0;
      // the dQ rows of a query chunk take a reduce-add from every
      // task of the chunk; a dK/dV tile one per bucket segment
      const uint64_t keep = l2_evict_last(), stream = l2_evict_first();
      for (uint32_t j = 0;; ++j) {
        if (kHoldReduce) break;
        const uint32_t slot = j % kInfo;
        if (!wait_bar_warp(sh, INFO_FULL + slot, (j / kInfo) & 1, a.status)) break;
        const TaskInfo& e = sh->info[slot];
        const int hi = e.hi, tok0 = e.tok0, kvrow = e.kvrow, flags = e.flags;
        const uint32_t seg = e.seg;
        __syncwarp();
        if (hi < 0) break;
        const uint32_t pb = j & 1;
        if (!wait_bar_warp(sh, DQ_FULL + pb, (j >> 1) & 1, a.status)) break;
        tc_fence_after();
        if constexpr (kDqFp32) {
          // fp32 dQ: four 32-dim pieces, each one 128-byte swizzled fp32 row
          // per lane of a 2-token x 16-head x 32-dim box
#pragma unroll 1
          for (int pc = 0; pc < 4; ++pc, ++chunk) {
            uint32_t v[32];
            tmem_ld32x(tmem + lane_base + col_dq(pb) + pc * 32, v);
            tmem_ld_wait();
            if (pc == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh->bar[DQ_EMPTY + pb]);
            }
            uint8_t* stg = stg0 + (chunk & 1) * 4096;
            if (lane == 0) bulk_wait_read_but_one();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                  make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_3d_hint(&tmdQ, stg, pc * 32, hi * 16, tok0 + 2 * sp, keep);
              bulk_commit();
            }
          }
        } else {
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf, ++chunk) {
            // 64 dims in two 32-column loads, each packed to bf16 on arrival
            uint32_t pq[32];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t v[32];
              tmem_ld32x(tmem + lane_base + col_dq(pb) + hf * 64 + h2 * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pq[h2 * 16 + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            }
            if (hf == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh->bar[DQ_EMPTY + pb]);
            }
            // 64 dims of this lane's row as bf16: one 128-byte swizzled row of a
            // 2-token x 16-head x 64-dim box
            uint8_t* stg = stg0 + (chunk & 1) * 4096;
            if (lane == 0) bulk_wait_read_but_one();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                  make_uint4(pq[4 * c], pq[4 * c + 1], pq[4 * c + 2], pq[4 * c + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_3d_hint(&tmdQ, stg, hf * 64, hi * 16, tok0 + 2 * sp, keep);
              bulk_commit();
            }
          }
        }
        if (flags & 2) {
          if (!wait_bar_warp(sh, DKV_FULL, seg & 1, a.status)) break;
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 4; ++q, ++chunk) {
            const int which = q >> 1, kh = q & 1;
            uint32_t v[32];
            const uint32_t col = (which ? COL_DV : COL_DK) + kh * 32;
            tmem_ld32(tmem + lane_base + col, v);
            if (q == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh->bar[DKV_EMPTY]);
            }
            uint8_t* stg = stg0 + (chunk & 1) * 4096;
            if (lane == 0) bulk_wait_read_but_one();
            __syncwarp();
#pragma unroll
            for (int ee = 0; ee < 32; ++ee)
              *reinterpret_cast<uint32_t*>(stg + ee * 128 + (((lane >> 2) ^ (ee & 7)) << 4) + (lane & 3) * 4) = v[ee];
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_3d_hint(which ? &tmdV : &tmdK, stg, sp * 32, 0, hi * a.W + kvrow + kh * 32, stream);
              bulk_commit();
            }
          }
        }
        // this reduce warp is done with the task: release its info entry
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->bar[INFO_EMPTY + slot]);
      }
      if (lane == 0) bulk_wait_all();
    }
  }
  __syncwarp();
  // drain: make sure no MMA is still writing TMEM before it is released (the
  // elected lane is the one that issued, the lowest lane of the warp)
  if (warp == kMmaWarp || warp == kMmaBWarp) {
    if (elect_one()) {
      umma_commit(&sh->bar[DRAIN]);
      wait_bar(sh, DRAIN, 0, a.status, false);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace msa
