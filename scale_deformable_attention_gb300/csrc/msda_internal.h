// msda_internal.h -- library-internal hooks shared between translation units
// (not part of the C ABI).
#pragma once

#include "../../include/msda.h"

namespace msda {
// Sets the calling thread's msda_last_error() message and returns `s`.
msda_status set_error(msda_status s, const char* message);
// Clears the calling thread's msda_last_error() message.
void clear_error();
}  // namespace msda
