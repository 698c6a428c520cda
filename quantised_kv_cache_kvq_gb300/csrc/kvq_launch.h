// kvq_launch.h -- host-side launchers shared between the translation units of libkvq.so.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kSmallAppend = 16;  // appends of at most this many tokens run as one kernel

int make_plan(const Layout& lo, DecodePlan* plan);
int device_sm_count(int device);
int decode_blocks(const void* fn, int threads, int64_t smem, int* nb);

int launch_append(const Layout& lo, uint8_t* cache, int layer, int seq_begin, int seq_count,
                  const void* k_new, const void* v_new, int n_new, const int32_t* n_valid,
                  const float* fp8_scales, uint32_t flags, cudaStream_t stream);
int launch_flush(const Layout& lo, uint8_t* cache, int layer, cudaStream_t stream);
int launch_decode(const Layout& lo, const DecodePlan& plan, const uint8_t* cache, int layer,
                  const void* q, float softmax_scale, float* out, uint8_t* ws, cudaStream_t stream);
int launch_lengths(const Layout& lo, const uint8_t* cache, int layer, int32_t* n_out,
                   int32_t* qn_out, cudaStream_t stream);

}  // namespace kvq
