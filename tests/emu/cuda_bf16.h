// Host stand-in for the bf16 header (CPU block emulator).
#pragma once
#include <cstdint>
struct __nv_bfloat16 {
  uint16_t x;
};
struct __nv_bfloat162 {
  uint16_t x, y;
};
