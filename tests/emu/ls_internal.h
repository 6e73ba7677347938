// Host stand-in for the library's internal header when one kernel's source
// is run on the CPU block emulator: the kernels need none of its host API.
#pragma once
#include <cuda_runtime.h>
