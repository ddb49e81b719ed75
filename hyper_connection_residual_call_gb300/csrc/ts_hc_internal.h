// ts_hc_internal.h -- host helpers that ts_hc_api.cu shares with the stack
// driver (ts_hc_stack.cu). Internal to the library.
#pragma once

#include "ts_hc.h"

namespace tshc {

// Clears the calling thread's last error.
void clear_error();
// Formats the calling thread's last error and returns `st`.
ts_status api_error(ts_status st, const char *fmt, ...);
// The shape rules every entry point shares (M >= 0, H, C, lowrank in range).
ts_status check_shape_api(int M, int H, int C, int lowrank);
// A device pointer that must be non-null and `align`-byte aligned.
ts_status check_ptr_api(const void *p, const char *name, size_t align);
// One hyper-connection module's tensors: hc_norm_w and the down / up weights,
// and the inject weight when `with_inject` (same format and group as down).
ts_status check_module(const ts_hc_module *m, bool with_inject, int H, int C, int lowrank,
                       const char *name);
// The PLE's shape rules (H a multiple of 128, C in range) and its module's tensors.
ts_status check_ple_shape(int H, int C);
ts_status check_ple_module(const ts_hc_ple_module *m);

}  // namespace tshc
