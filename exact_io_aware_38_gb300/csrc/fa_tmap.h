// Host-side TMA tensor maps for [B*H][N][D] bf16 tensors (3-D view, boxes of 64 columns x
// `box_rows` rows, 128-byte swizzle). Rows past N in a head read as zero and are never written.
#pragma once

#include <cuda.h>

bool fa_make_tmap_bf16(CUtensorMap* m, const void* ptr, int N, int D, int BH, int box_rows = 128);
