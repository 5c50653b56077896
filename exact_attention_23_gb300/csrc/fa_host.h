// Host-side helpers shared by the forward (fa_api.cu) and backward (fa_bwd_api.cu) entry
// points. Internal; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace fa {
namespace host {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder (looked up once), or null.
EncodeTiledFn encode_fn();
// FA_OK with the current device and its SM count if it is compute capability 10.3.
int check_device(int* dev_out, int* sms_out);
// 3-D map over a [B·H][T][d] bf16 tensor, boxes of 64 columns × box_rows rows × 1 head.
bool encode_map(EncodeTiledFn enc, CUtensorMap* map, const void* base, int T, int d, int BH,
                int box_rows = 128);
bool overlaps(const void* a, size_t na, const void* b, size_t nb);
// A softmax factor the kernels can take: finite, and so is scale·log2(e) in fp32 (every
// sign and zero included).
bool scale_ok(float scale);
// The tensor-core kernels' exponent factor for scale·log2(e) = sl2: they take the row
// maximum of S before multiplying by the factor, so the factor must be positive. sl2 < 0
// runs as S = −Q·Kᵀ (the S product's A-negate bit, *negate) with factor −sl2; sl2 = 0 runs
// with the smallest normal float, under which every score s with |s| < 2^102 gives
// exactly 2^(s·c − m) = 1 (uniform weights) and masked scores still give 0.
float exponent_factor(double sl2, unsigned* negate);
bool aligned16(const void* p);

}  // namespace host
}  // namespace fa
