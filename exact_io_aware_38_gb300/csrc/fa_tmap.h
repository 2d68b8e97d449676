// Host-side TMA tensor maps for [B*H][N][D] bf16 tensors (3-D view, 64 x 128 boxes, 128-byte
// swizzle). Rows past N in a head read as zero and are never written.
#pragma once

#include <cuda.h>

bool fa_make_tmap_bf16(CUtensorMap* m, const void* ptr, int N, int D, int BH);
