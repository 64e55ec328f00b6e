// Tiling of the split-K router GEMV with last-arriver fixup, used for
// 64 < M <= 512 (the pages tune BLOCK_N and SPLIT_K per M bucket, sglang
// #36557 description; M <= 64 runs the cluster kernel of route_kernel.cuh).
//   X(index, MT, HALF, NW, KW, KS)
//   MT   16-row tiles per CTA     HALF  only rows 0..7 live (M <= 8)
//   NW   8-expert tiles per CTA   KW    warps along K   KS  32-wide k steps per warp
// BLOCK_N = 8*NW, K per CTA = 32*KS*KW, threads = 32*NW*KW.
#pragma once

#define MR_GEMV_CONFIGS(X) \
    X(0, 4, false, 2, 4, 2)

// Bucket -> table row (64-row tiles).
#define MR_GEMV_CFG_ROWS64 0
