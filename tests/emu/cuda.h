// Host stand-in for the CUDA driver header (CPU block emulator): a tensor
// map is the emulator's record of the encoded tiled map.
#pragma once
#include "emu_core.h"
typedef emu::TensorMap CUtensorMap;
