// Host-side TMA tensor maps for bf16 tensors addressed as [batch][row][head][d] with arbitrary
// element strides (4-D view d, rows, heads, batches; boxes of 64 columns x `box_rows` rows of one
// head, 128-byte swizzle). Rows past `rows` read as zero and are never written.
#pragma once

#include <cuda.h>

bool fa_make_tmap_bf16(CUtensorMap* m, const void* ptr, int D, int rows, int heads, int batches, long long row_stride,
                       long long head_stride, long long batch_stride, int box_rows = 128);
