// Host-side helpers shared by the translation units of the MSA library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/msa.h"

namespace msa {

constexpr int kHeadDim = 128;
// Key tile of the backward and forward kernels: a 64-key block is one tile,
// a 128-key block two.
constexpr int kKeyTile = 64;
constexpr int kChunk = 8;
constexpr int kGroup = 16;
constexpr int kMaxTopk = 32;
// Largest number of key-block rows a problem may have (3M tokens of 64-key
// blocks): keeps the CSR build's per-group row counters, index heads x groups
// x rows of int32, to a few hundred MB and every offset inside int32.
constexpr int kMaxRows = 49152;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Host-checkable problem validity (shapes the kernels are built for).
int check_problem(const msa_problem* p);

// Scatter-group size (query chunks per group) of the CSR build.
inline int64_t k2q_group_chunks(int64_t nc) {
  int64_t g = (nc + 127) / 128;
  return g < 64 ? 64 : g;
}
inline int key_tiles_per_block(const msa_problem* p) { return p->block_size / kKeyTile; }
inline int64_t num_tiles(int64_t nc, int32_t tile_chunks) {
  return tile_chunks > 0 ? (nc + tile_chunks - 1) / tile_chunks : 1;
}

size_t k2q_ws_bytes(const msa_problem* p);
size_t select_ws_bytes(const msa_problem* p);
// Launches the document-layout kernel: blk_off[d], chunk_off[d] for d in
// [0, N] (device int32 [N+1] each) and the consistency checks of cu_seqlens
// and kv_doc_starts (MSA_ERR_INVALID_DOCUMENTS in *status).
int launch_layout(const msa_problem* p, int32_t* blk_off, int32_t* chunk_off, int32_t* status, cudaStream_t st);
size_t tasks_ws_bytes(const msa_problem* p, int32_t tile_chunks);
size_t bwd_ws_bytes(const msa_problem* p, bool dq_fp32);

int sm_count_current(int32_t* out);
int check_device_current();

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

}  // namespace msa
