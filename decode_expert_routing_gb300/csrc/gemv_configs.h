// Per-M-bucket tiling of the router GEMV (the pages tune BLOCK_N and SPLIT_K
// per bucket M <= 8 / 16 / 32 / 64, sglang #36557 description; these rows
// are this library's own, for GB300).
//   X(index, MT, HALF, NW, KW, KS)
//   MT   16-row tiles per CTA     HALF  only rows 0..7 live (M <= 8)
//   NW   8-expert tiles per CTA   KW    warps along K   KS  32-wide k steps per warp
// BLOCK_N = 8*NW, K per CTA = 32*KS*KW, threads = 32*NW*KW.
#pragma once

#define MR_GEMV_CONFIGS(X)       \
    X(0, 1, true, 2, 4, 4)       \
    X(1, 1, false, 2, 4, 4)      \
    X(2, 2, false, 2, 4, 2)      \
    X(3, 4, false, 2, 4, 2)

// Bucket -> table row.
#define MR_GEMV_CFG_M8 0
#define MR_GEMV_CFG_M16 1
#define MR_GEMV_CFG_M32 2
#define MR_GEMV_CFG_M64 3
