// pkd_tc_launch.h -- host entry of the tcgen05 decode kernel (pkd_inst_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include "pkd_decode.cuh"

namespace pkd {

// Query rows (query tokens x group heads) one CTA of the tcgen05 kernel serves.
constexpr int kTcRowsPerCta = 64;

// Launch `grid` CTAs of the tcgen05 kernel; p.q_chunks must be
// ceil(q_len / (kTcRowsPerCta / G)).  kvb: bytes per cache element (2: fp16;
// 1: E4M3, with p.scale_log2 including the K scale and p.v_scale the V scale).
// head_dim 128, or 64 with fp16 caches; block size 16 or 32
// (cudaErrorInvalidValue otherwise).
cudaError_t launch_decode_tcgen05(int D, int BS, const DecodeParams& p, long long grid, cudaStream_t stream,
                                  int kvb = 2);

}  // namespace pkd
