// msda_internal.h -- library-internal hooks shared between translation units
// (not part of the C ABI).
#pragma once

#include "../../include/msda.h"

namespace msda {
// Sets the calling thread's msda_last_error() message and returns `s`.
msda_status set_error(msda_status s, const char* message);
// Clears the calling thread's msda_last_error() message.
void clear_error();
// Bytes of workspace the FP32 accumulator runs with for fp16/bf16 I/O: the
// fp32 sums (B*S*M*D*4, or the on-chip accumulator's smaller layout when
// MSDA_TUNE selects it), plus the touch classes of their rows with `touch`.
size_t fp32_workspace_bytes(msda_dtype dt, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, int64_t K,
                            int64_t Q, bool touch);
}  // namespace msda
