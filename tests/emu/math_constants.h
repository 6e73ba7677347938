// Host stand-in for CUDA's math constants (CPU block emulator).
#pragma once
#include <cmath>
#define CUDART_INF_F INFINITY
