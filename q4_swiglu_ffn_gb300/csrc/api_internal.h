// Services of api.cu that the other entry-point files of the library use
// (library-internal, not part of the C ABI).
#pragma once
#include <stdint.h>

#include "q4kffn.h"

namespace q4k {

// Checks (once per device) that the current device is an sm_103 part and
// returns its SM count and the device address of the library's error word.
// Allocates nothing.
q4k_status current_device(int* sms, uint32_t** err);

// Resolves x and y as the FFN entry points do: device or managed memory is used
// as is, mapped page-locked host memory is replaced by its device address, and
// anything else (pageable or unmapped host memory) gives Q4K_ERR_MEMORY.
q4k_status resolve_host_io(const void** x, float** y);

// Records a failed host-side call for q4k_get_last_error() on this thread and
// returns the status.
q4k_status record_failure(q4k_status s);

// Records the number of kernels the call launched, for q4k_last_call_kernels().
void record_kernels(int n);

}  // namespace q4k
