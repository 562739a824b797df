// CTA tilings compiled for each kernel family: X(R, WN, WK).
//   mma:  R 16-row tiles per warp, WN warps along N, WK warps along K.
#pragma once

#define QMM_MMA_TILES(X) \
  X(2, 2, 4)             \
  X(1, 2, 4)             \
  X(4, 1, 8)

//   tma:  X(W consumer warps, maximum ring stages)
#define QMM_TMA_TILES(X) \
  X(8, 16)               \
  X(4, 16)               \
  X(16, 16)

//   own:  X(W consumer warps, ring stages per warp)
#define QMM_OWN_TILES(X) \
  X(8, 3)                \
  X(16, 2)               \
  X(4, 4)                \
  X(8, 2)
