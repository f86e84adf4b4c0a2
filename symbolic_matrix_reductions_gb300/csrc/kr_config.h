// kr_config.h -- compile-time shapes of the kernel instances, shared by the host
// planner and the device code (constexpr, no CUDA dependency).
#pragma once

#ifdef __CUDACC__
#define KR_HD __host__ __device__
#else
#define KR_HD
#endif

namespace kr {

// Coordinate count the instance is compiled for: exact for D <= 4, else the next
// of 8, 16, 32, 50, 64, 128 (padded coordinates are zero on both sides, so they
// add nothing to a distance).
KR_HD constexpr int pad_d(int D) {
    return D <= 4 ? D : D <= 8 ? 8 : D <= 16 ? 16 : D <= 32 ? 32 : D <= 50 ? 50 : D <= 64 ? 64 : 128;
}
// Signal columns the instance is compiled for (zero-padded signal columns).
KR_HD constexpr int pad_e(int E) { return E <= 1 ? 1 : E <= 4 ? 4 : 16; }
// K-min list length the instance keeps (the first K of a longer sorted list are
// the K smallest).
KR_HD constexpr int pad_k(int K) { return K <= 1 ? 1 : K <= 4 ? 4 : K <= 10 ? 10 : K <= 16 ? 16 : 32; }

// Floats per point in the shared-memory tile: coordinates then values, rounded
// up to whole float4s so every point is read with 16-byte loads.
KR_HD constexpr int pack_stride(int DP, int VP) { return (DP + VP + 3) / 4 * 4; }

// Points of y per tile: the largest power of two whose tile fits in 32 KB,
// between 32 and 512.
KR_HD constexpr int tile_points(int PS) {
    return (8192 / PS) >= 512 ? 512 : (8192 / PS) >= 256 ? 256 : (8192 / PS) >= 128 ? 128
         : (8192 / PS) >= 64 ? 64 : 32;
}

// Rows of x each thread keeps in registers (each shared-memory read of y_j then
// feeds R pairs).  Chosen so that coordinates, accumulators and the K-min list
// stay in registers.
KR_HD constexpr int rows_fwd(int DP, int EP) {
    return EP >= 16 ? 1 : EP >= 4 ? (DP <= 8 ? 2 : 1) : (DP <= 8 ? 4 : DP <= 16 ? 2 : 1);
}
KR_HD constexpr int rows_grad(int DP, int EP) {
    return DP <= 4 ? (EP == 1 ? 4 : EP == 4 ? 2 : 1) : DP <= 8 ? (EP == 1 ? 2 : 1) : 1;
}
KR_HD constexpr int rows_knn(int DP, int KP) {
    return DP <= 16 ? (KP <= 10 ? 4 : 2) : 1;
}

// Tensor-core Sum: largest |x'|^2 + |y'|^2 (prescaled, base-2 exponent units) for
// which the expanded exponent 2x'.y' - |x'|^2 - |y'|^2, accumulated in fp32 from
// split fp16 operands, keeps the kernel values within the Sum tolerance (its
// absolute error is a few 1e-6 times this sum).
constexpr float kTcNormLimit = 16.0f;
// Tensor-core Sum geometry: rows per block (TMEM lanes, MMA M), points per tile
// (MMA N), threads per block (a TMA warp, an MMA warp, 8 evaluation warps).
constexpr int kTcRows = 128;
constexpr int kTcCols = 256;
constexpr int kTcThreads = 320;
// Coordinate range of the tensor-core Sum (the augmented vector must fit K = 64).
KR_HD constexpr bool tc_dims(int D, int E) { return E == 1 && D >= 32 && D <= 62; }
// The tensor-core LogSumExp adds the tile-relative log-weight as one more slot.
constexpr int kTcLseMaxD = 61;
// Tensor-core x-gradient: points per tile (the N of its first product and the K of its
// second, P . [y' | 1]); same coordinate range as the Sum (the second product reads the
// augmented B tile, whose slot D holds 1).
constexpr int kTcGradCols = 128;
// Tensor-core K-min screen: rows per block (two A tiles of kTcRows, each its own MMA M) and
// points per tile (MMA N), so that every B tile read from L2 serves 256 rows.
constexpr int kTcKnnRows = 256;
constexpr int kTcKnnCols = 128;

// Independent partial sums of a squared distance: at large D one fma chain over the
// coordinates is a long dependency chain (4 cycles a link) with few rows per thread to
// hide it, so the sum is split into this many interleaved chains, added at the end.
KR_HD constexpr int dist_chains(int DP) { return DP >= 32 ? 4 : DP >= 16 ? 2 : 1; }
// Inner-loop unroll over tile points (tiles are padded to a multiple of it).
KR_HD constexpr int unroll_points(int DP) { return DP <= 8 ? 4 : DP <= 32 ? 2 : 1; }

// Packed (f32x2) instances evaluate two points per instruction; they keep x'
// duplicated in register pairs, so they are used up to D = 64.
KR_HD constexpr bool packed(int DP) { return DP <= 64; }
// The packed gradient also keeps 2 R D partial sums in registers: up to D = 16.
KR_HD constexpr bool packed_grad(int DP) { return DP <= 16; }
// Wide gradient (32 <= D <= 64): one row per thread with x, the differences and the
// tile's partial sums in registers (3 D floats) and the compensated running sums in
// shared memory, so the block needs no more than ~170 registers a thread.
KR_HD constexpr bool wide_grad(int DP) { return DP >= 32 && DP <= 64; }
// Points per tile of the wide gradient (the tile and the running sums share the
// block's dynamic shared memory).
constexpr int kWideGradTile = 64;
// Pair record: points 2m and 2m+1 of a tile interleaved field by field, so one
// 16-byte load yields two float2 operands; rounded up to whole float4s.
KR_HD constexpr int pair_stride(int DP, int VP) { return (2 * (DP + VP) + 3) / 4 * 4; }
// Points per tile for pair records: a power of two, at most 512, tile <= 32 KB.
KR_HD constexpr int tile_points_packed(int PS2) {
    return (16384 / PS2) >= 512 ? 512 : (16384 / PS2) >= 256 ? 256 : (16384 / PS2) >= 128 ? 128
         : (16384 / PS2) >= 64 ? 64 : 32;
}
// Streamed records (Gaussian Sum, LogSumExp and x-gradient up to D = 16): a prepass packs
// the call's y (prescaled and negated) and its signal (or the LogSumExp's tile-relative
// log-weight) once into tile-aligned pair records in device memory, and the reduction
// kernel copies each tile into shared memory with 16-byte cp.async, double-buffered, so
// the next tile's copy overlaps the current tile's scan and a tile costs one barrier.
// Batched calls (many small problems) keep the kernels' own staging.
KR_HD constexpr bool streamed(int DP) { return DP <= 16; }
// Floats of one tile of pair records (BN points).
KR_HD constexpr int record_tile_floats(int DP, int EP, int BN) { return (BN / 2) * pair_stride(DP, EP); }
// Filtered K-min: the pass bits of this many consecutive point groups are gathered in one
// word per row and queued as one entry (block index, bit mask), so the scan loop itself
// carries no branch.
KR_HD constexpr int knnx_mask_groups(int DP, int KP) { return 8; }
// Entries per row of the filtered K-min's queue (0: immediate insertion).
KR_HD constexpr int knnx_queue(int DP, int KP) { return DP <= 16 ? 8 : 0; }
// Resident blocks per SM the K-min instances are compiled for (registers cap): the
// queued filtered instances keep at most 128 (D <= 4, K <= 16), 170 (D = 8, K = 16) or
// 255 registers (four rows at D = 8 or 16, or two rows of 32-entry lists).  At D = 8
// and 16 the screen's records are wide (20 and 36 floats a point pair), so four rows
// per record read are worth the lower occupancy: the loop is bound by shared memory.
KR_HD constexpr int knn_min_blocks(int DP, int KP) {
    return knnx_queue(DP, KP) > 0 ? (DP <= 4 ? (KP <= 16 ? 4 : 2) : DP <= 8 ? (KP == 16 ? 3 : 2) : 2) : 1;
}
// Pair records per unrolled step of the packed inner loop.
KR_HD constexpr int unroll_pairs(int DP) { return DP <= 8 ? 2 : 1; }
// Tile points of an instance (value columns VP = E, K-min: 0).
KR_HD constexpr int instance_tile(int DP, int VP) {
    return packed(DP) ? tile_points_packed(pair_stride(DP, VP)) : tile_points(pack_stride(DP, VP));
}

// K-min with the expansion filter: |y~|^2 - 2 x~.y~ (D FMAs a pair) screens groups of
// points and only the groups that may hold a candidate get the direct distance.  Used
// up to D = 16, where a tile record is shared by 2-4 rows of a thread and its
// shared-memory loads stay well below the FMA work; at larger D one row per thread
// would make the loop load-bound.
KR_HD constexpr bool knn_expand(int DP) { return DP <= 16; }
// Margin of the filter per unit of |x~|^2 + |y~|^2 + threshold: (8 DP + 12) u with
// u = 2^-24, twice the first-order bound on the rounding the filter can hide.
KR_HD constexpr float knn_kappa(int DP) { return (float)(8 * DP + 12) * 5.9604644775390625e-8f; }
// Tile points of the filtered K-min: its two record arrays (filter: -y~ and h; exact:
// -y) together within 36 KB of static shared memory.  Up to 1024 points: the queues
// are drained at least once a tile, and a longer tile gives each lane more entries
// per drain, so the warp-wide drain steps are better filled.
KR_HD constexpr int knn_tile_bytes(int DP, int BN) { return (BN / 2) * (pair_stride(DP, 1) + pair_stride(DP, 0)) * 4; }
KR_HD constexpr int knn_tile(int DP) {
    return knn_tile_bytes(DP, 1024) <= 36864 ? 1024 : knn_tile_bytes(DP, 512) <= 36864 ? 512
         : knn_tile_bytes(DP, 256) <= 36864 ? 256 : knn_tile_bytes(DP, 128) <= 36864 ? 128 : 64;
}
// Tile points of the K-min instance for DP.
KR_HD constexpr int knn_instance_tile(int DP) { return knn_expand(DP) ? knn_tile(DP) : instance_tile(DP, 0); }

}  // namespace kr
