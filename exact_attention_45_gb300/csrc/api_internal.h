// api_internal.h -- helpers the C-ABI translation units share (not exported).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn45 {
int api_fail(int code, const char* msg);
int api_cuda_fail(cudaError_t e, const char* what);
unsigned long long api_timeout_ns();
// Current device: checks it is a GB300 and returns its SM count and the
// device error word.
int api_device(int* sm_count, unsigned int** err);
// 4-D tiled tensor map {inner, heads, rows, batch}, box {box_inner, 1,
// box_rows, 1}, 128-byte swizzle, zero fill out of bounds; u8 or bf16 data.
int api_make_map(CUtensorMap* m, bool u8, const void* base, uint64_t inner, uint64_t heads, uint64_t rows,
                 uint64_t batch, uint32_t box_inner, uint32_t box_rows);
// u8 tensor [batch][rows][inner] as a 4-D map {inner, rows, batch, 1} with box
// {box_inner, box_rows, 1, 1}, 128-byte swizzle.
int api_make_map_rows(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t batch,
                      uint32_t box_inner, uint32_t box_rows);
}  // namespace attn45
