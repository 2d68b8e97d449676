// Host-side TMA tensor maps for bf16 tensors addressed as [batch][row][head][d] with arbitrary
// element strides (4-D view d, rows, heads, batches; boxes of 64 columns x `box_rows` rows of one
// head, 128-byte swizzle). Rows past `rows` read as zero and are never written.
#pragma once

#include <cuda.h>

bool fa_make_tmap_bf16(CUtensorMap* m, const void* ptr, int D, int rows, int heads, int batches, long long row_stride,
                       long long head_stride, long long batch_stride, int box_rows = 128);
// The same for 8-bit elements (e4m3 operands) with a box of box_inner elements (bytes) x box_rows;
// strides in bytes. box_inner * 1 byte must not exceed the 128-byte swizzle span.
bool fa_make_tmap_u8(CUtensorMap* m, const void* ptr, int inner, int rows, int heads, int batches, long long row_stride,
                     long long head_stride, long long batch_stride, int box_inner, int box_rows);
