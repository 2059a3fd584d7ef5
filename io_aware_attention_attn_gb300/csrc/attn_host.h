// attn_host.h -- host-side helpers shared by the C-ABI entry points (not part of the public API).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

// Encode a 3-D TMA map over a [heads][rows][d] bf16 tensor (d innermost) with a
// {64, box_rows, 1} box and 128-byte swizzle: one box is a box_rows x 64-column block
// (16 KB for 128 rows), the shared-memory layout the tcgen05 descriptors expect.  Rows past
// `rows` read as zero.  Returns a CUresult.
int encode_rows_map(CUtensorMap* map, const void* base, uint64_t d, uint64_t rows,
                    uint64_t heads, uint32_t box_rows = 128);

// Same for an fp32 [heads][rows][cols] tensor with a {32, 128, 1} box (128-byte rows, swizzled).
int encode_f32_rows_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                        uint64_t heads);

// 0 if the current device is sm_103 (checked once per device), else an attn_status code.
int check_device();

// Device address of the status word on the current device (nullptr on failure).
int* status_word();

}  // namespace attn
