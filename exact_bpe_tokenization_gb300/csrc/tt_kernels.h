// tt_kernels.h - host-side launchers of the tokenizer's kernels.
#pragma once
#include <cuda_runtime.h>

#include "tt_common.cuh"

namespace tt {

cudaError_t pretok_configure();
cudaError_t bpe_configure();
void launch_prepass(const Tables &T, const Work &W, int grid, cudaStream_t s);
void launch_pretok(const Tables &T, const Work &W, int grid, cudaStream_t s);

void launch_lit_find(const Tables &T, const Work &W, int grid, cudaStream_t s);
void launch_lit_pick(const Tables &T, const Work &W, int grid, cudaStream_t s);
void launch_bpe_warp(const Tables &T, const Work &W, int grid, cudaStream_t s);
void launch_bpe_long(const Tables &T, const Work &W, int grid, cudaStream_t s);
void launch_idscan(const Work &W, cudaStream_t s);
void launch_ids(const Tables &T, const Work &W, int grid, cudaStream_t s);

void launch_hook_pre(const Work &W, cudaStream_t s);
void launch_hook_pieces(const Work &W, int grid, cudaStream_t s);
void launch_hook_offsets(const Work &W, int grid, cudaStream_t s);

constexpr int BPE_WARP_THREADS = 256;
constexpr int BPE_WARP_CTAS_PER_SM = 4;   // all resident: 64 registers, 32 KB shared memory each
constexpr int BPE_LONG_THREADS = 512;
constexpr int IDS_THREADS = 256;

}  // namespace tt
