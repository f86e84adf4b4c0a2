// kr_tc.cu -- tensor-core (tcgen05) path of the Gaussian Sum, LogSumExp and x-gradient
// for 32 <= D <= 62, E = 1 (the x-gradient's two products are described at its kernel).
//
// The exponent of the prescaled Gaussian is a dot product of augmented vectors:
//   -|x' - y'|^2 = 2 x'.y' - |x'|^2 - |y'|^2 = A_i . B_j,
//   A_i = [2 x'_i, -|x'_i|^2, -1, 0...],  B_j = [y'_j, 1, |y'_j|^2, 0...]   (K = 64),
// so a 128-row block of A against a 256-point tile of B is one M=128, N=256, K=64
// matrix product on the 5th-generation tensor cores, accumulated in fp32 in tensor
// memory (TMEM).  fp16 operands alone would carry 11 bits; each value v is split
// as v = hi + lo (both fp16, lo = fp16(v - hi)) and the product is taken as
// hi.hi + hi.lo + lo.hi (12 MMAs of K = 16): the dropped lo.lo term and the
// split residual are below 2^-21 |v|.  The expansion cancels |x'|^2 + |y'|^2 down to
// -|x'-y'|^2, so its absolute error grows with the norms: a prepass records the
// largest |x'|^2 and |y'|^2 and, when their sum exceeds kTcNormLimit, the tensor
// kernel leaves the work to the CUDA-core kernel launched after it (which runs only
// in that case), without a host round trip.
//
// The LogSumExp (tc_lse_kernel) adds the weight to the product itself: the prepass
// gives A one more slot of 1 and B the point's log-weight relative to its tile's
// largest, w' - F (w' = w log2 e, at least -1024, so an empty weight is a term of 0),
// so the accumulator already holds t + w' - F <= 0 (t <= 0 is the exponent above) and
// the evaluation reads nothing but TMEM; the warps fold each tile's partial into a
// running (frame, hi, lo) per row.  Within the norm guard t >= -32, so the tile's
// largest-weight term is at least 2^-32 and the partial cannot vanish while a finite
// weight is present.  The split fp16 pair carries w' - F to 2^-21 of its size, and
// a term whose w' - F is large is negligible beside the tile's largest.
//
// Block = 10 warps, one block per SM, warp-specialised around mbarriers:
//   warp 0, one thread: TMA producer.  Loads the block's A tiles (hi, lo) once, then
//     streams B tiles of 256 points (hi, lo: 2 x 32 KB, landing in the
//     128-byte-swizzled K-major layout the MMA reads) into a ring of kStages stages.
//   warp 1: allocates TMEM; one thread issues the 12 MMAs (M=128, N=256, K=16) of
//     each tile into one of two TMEM accumulators of 256 columns and commits them to
//     the stage's `empty` barrier and the accumulator's `full` barrier.  A tcgen05
//     MMA runs 128 x 256 x 16 in 128 cycles, but every barrier poll or commit
//     between MMAs lets the MMA queue run dry for about 100 cycles, so the tiles are
//     as wide as TMEM allows: 12 MMAs per handshake.
//   warps 2-9: evaluation.  Warp w reads TMEM lanes 32 (w mod 4)..+31 (its rows);
//     warps w and w+4 take the two 128-column halves of the tile.  Each loads its
//     half, releases the accumulator (the MMAs of tile i+2 may then overwrite it),
//     computes 2^t and accumulates b_j 2^t.  The Sum loads in the 16x256b shape (a
//     thread holds 4 rows x 32 columns), so a thread reads b at 32 columns only (the
//     prepass stores them contiguously; L1 broadcasts) and adds column pairs with
//     f32x2 FMAs; the four lanes that share rows are combined at the end.  The
//     LogSumExp loads one row per lane (32x32b) and reads nothing else.
// Every mbarrier wait is bounded (by global time, default 2 s, and a poll count); a
// role that gives up raises a block-wide abort flag, and every role then leaves its
// loop; the producer and the MMA issuer then wait (bounded) for their copies and MMAs
// in flight, the block's rows come out as NaN, and bit 0 of a sticky device status
// word is set, which kr_device_status() reads and clears.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kr_kernels.cuh"
#include "kr_tc.h"

namespace kr {

namespace {

constexpr int kRows = kTcRows;          // rows per block = TMEM lanes = MMA M
constexpr int kCols = kTcCols;          // points per tile = MMA N
constexpr int kStages = 3;              // B tiles in flight
constexpr int kEvalWarps = 8;           // two per TMEM lane quarter
constexpr int kEvalCols = kCols / 2;    // tile columns per evaluation warp
constexpr int kThreadsTc = kTcThreads;
constexpr int kATileBytes = kRows * 128;  // 128 rows x 64 fp16
constexpr int kBTileBytes = kCols * 128;  // 256 rows x 64 fp16
constexpr int kTmemCols = 2 * kCols;      // two fp32 accumulators
constexpr long kWaitLimit = 1L << 26;     // mbarrier polls before giving up
static_assert(kThreadsTc == 64 + 32 * kEvalWarps, "warp roles");
static_assert(kCols == 256, "the prepass computes an LSE tile frame per block of 256 threads");
static_assert(kTmemCols <= 512, "TMEM has 512 columns");

// Dynamic shared memory: A hi, A lo, kStages x (B hi, B lo), plus 1 KB of alignment
// slack (the 128-byte swizzle wants 1024-byte aligned tiles).
constexpr int kStageBytes = 2 * kBTileBytes;
constexpr int kSmemBytes = 2 * kATileBytes + kStages * kStageBytes + 1024;
static_assert(kSmemBytes + 256 <= 227 * 1024, "shared memory per block");

// tcgen05 instruction descriptor: D = f32, A = B = f16, both K-major, M = kRows (128),
// N = kCols (256).
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kCols >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 bytes,
// 8-row (1024-byte) swizzle atoms, so the stride between 8-row groups is 1024 B.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// The same tile read MN-major (the gradient's second product reads the B tile's point
// rows as its K dimension): N = 64 fp16 is one 128-byte swizzle row, so only the stride
// between 8-row groups along K matters (1024 B); the other byte offset is given the same
// value, so it is right whichever of the two fields the layout takes it from.
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)(1024 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// The descriptor of base + off from the base's: the start address (16-byte units, bits
// 0-13) is the low field of the low word, and a block's shared memory stays below 256 KB,
// so off / 16 adds to the low word without carrying out of the field.  One integer add an
// operand, for issue loops that place many products in the same tiles.
__device__ __forceinline__ uint64_t desc_add(uint64_t base, uint32_t off) {
    return (base & 0xFFFFFFFF00000000ull) | (uint64_t)((uint32_t)base + (off >> 4));
}

// D[tmem] (+)= A[smem] . B[smem]^T, fp16 operands, fp32 accumulation (instruction
// descriptor idesc: shapes and operand majors).
__device__ __forceinline__ void mma_f16(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t accumulate,
                                        uint32_t idesc = kIdesc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
        "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the completion of the phase with the given parity.  Gives up
// (raising `abort`) after `limit_ns` of global time or kWaitLimit polls, whichever
// comes first, or early when another role raised `abort`.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, volatile int *abort, uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (long it = 0; it < kWaitLimit; ++it) {
        if (mbar_try(mbar, parity)) return true;
        if ((it & 255) == 255) {
            if (*abort) return false;
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > limit_ns) break;
        }
    }
    *abort = 1;
    return false;
}

// Bounded wait that ignores `abort`: used after an abort, to let this block's own
// copies and MMAs in flight land before the block releases its memory.
__device__ __forceinline__ bool mbar_drain(uint32_t mbar, uint32_t parity, uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (long it = 0; it < kWaitLimit; ++it) {
        if (mbar_try(mbar, parity)) return true;
        if ((it & 255) == 255) {
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > limit_ns) break;
        }
    }
    return false;
}

// Sticky device-side status of the tensor-core kernels: bit 0 = a bounded wait gave up
// (the rows of that block came out NaN).  Read and cleared by tc_read_status().
__device__ unsigned int g_tc_status;

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(mbar)
        : "memory");
}

// One warp reads 128 consecutive fp32 columns of 16 TMEM lanes (from lane base B) in
// the 16x256b shape: register 4k + 2h + e of thread t holds lane B + t/4 + 8h, column
// 8k + 2(t%4) + e (k < 16; h, e < 2).
__device__ __forceinline__ void tmem_ld16x256_x16(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31]),"=r"(r[32]),"=r"(r[33]),"=r"(r[34]),"=r"(r[35]),"=r"(r[36]),"=r"(r[37]),"=r"(r[38]),"=r"(r[39]),"=r"(r[40]),"=r"(r[41]),"=r"(r[42]),"=r"(r[43]),"=r"(r[44]),"=r"(r[45]),"=r"(r[46]),"=r"(r[47]),"=r"(r[48]),"=r"(r[49]),"=r"(r[50]),"=r"(r[51]),"=r"(r[52]),"=r"(r[53]),"=r"(r[54]),"=r"(r[55]),"=r"(r[56]),"=r"(r[57]),"=r"(r[58]),"=r"(r[59]),"=r"(r[60]),"=r"(r[61]),"=r"(r[62]),"=r"(r[63])
                 : "r"(taddr));
}

// One warp reads 128 consecutive fp32 columns of its 32 TMEM lanes (one row per lane).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];"
                 : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31]),"=r"(r[32]),"=r"(r[33]),"=r"(r[34]),"=r"(r[35]),"=r"(r[36]),"=r"(r[37]),"=r"(r[38]),"=r"(r[39]),"=r"(r[40]),"=r"(r[41]),"=r"(r[42]),"=r"(r[43]),"=r"(r[44]),"=r"(r[45]),"=r"(r[46]),"=r"(r[47]),"=r"(r[48]),"=r"(r[49]),"=r"(r[50]),"=r"(r[51]),"=r"(r[52]),"=r"(r[53]),"=r"(r[54]),"=r"(r[55]),"=r"(r[56]),"=r"(r[57]),"=r"(r[58]),"=r"(r[59]),"=r"(r[60]),"=r"(r[61]),"=r"(r[62]),"=r"(r[63]),"=r"(r[64]),"=r"(r[65]),"=r"(r[66]),"=r"(r[67]),"=r"(r[68]),"=r"(r[69]),"=r"(r[70]),"=r"(r[71]),"=r"(r[72]),"=r"(r[73]),"=r"(r[74]),"=r"(r[75]),"=r"(r[76]),"=r"(r[77]),"=r"(r[78]),"=r"(r[79]),"=r"(r[80]),"=r"(r[81]),"=r"(r[82]),"=r"(r[83]),"=r"(r[84]),"=r"(r[85]),"=r"(r[86]),"=r"(r[87]),"=r"(r[88]),"=r"(r[89]),"=r"(r[90]),"=r"(r[91]),"=r"(r[92]),"=r"(r[93]),"=r"(r[94]),"=r"(r[95]),"=r"(r[96]),"=r"(r[97]),"=r"(r[98]),"=r"(r[99]),"=r"(r[100]),"=r"(r[101]),"=r"(r[102]),"=r"(r[103]),"=r"(r[104]),"=r"(r[105]),"=r"(r[106]),"=r"(r[107]),"=r"(r[108]),"=r"(r[109]),"=r"(r[110]),"=r"(r[111]),"=r"(r[112]),"=r"(r[113]),"=r"(r[114]),"=r"(r[115]),"=r"(r[116]),"=r"(r[117]),"=r"(r[118]),"=r"(r[119]),"=r"(r[120]),"=r"(r[121]),"=r"(r[122]),"=r"(r[123]),"=r"(r[124]),"=r"(r[125]),"=r"(r[126]),"=r"(r[127])
                 : "r"(taddr));
}

// One warp reads n consecutive fp32 columns of its 32 TMEM lanes (one row per lane).
__device__ __forceinline__ void tmem_ld32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31]),"=r"(r[32]),"=r"(r[33]),"=r"(r[34]),"=r"(r[35]),"=r"(r[36]),"=r"(r[37]),"=r"(r[38]),"=r"(r[39]),"=r"(r[40]),"=r"(r[41]),"=r"(r[42]),"=r"(r[43]),"=r"(r[44]),"=r"(r[45]),"=r"(r[46]),"=r"(r[47]),"=r"(r[48]),"=r"(r[49]),"=r"(r[50]),"=r"(r[51]),"=r"(r[52]),"=r"(r[53]),"=r"(r[54]),"=r"(r[55]),"=r"(r[56]),"=r"(r[57]),"=r"(r[58]),"=r"(r[59]),"=r"(r[60]),"=r"(r[61]),"=r"(r[62]),"=r"(r[63])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31])
                 : "r"(taddr));
}

__device__ __forceinline__ bool norms_ok(const unsigned *guard) {
    return __uint_as_float(guard[0]) + __uint_as_float(guard[1]) <= kTcNormLimit;
}

// The power of two 2^e >= m (m >= 0 finite; 1 for m = 0): the x-gradient scales its signal
// by 2^-e into [-1, 1], which keeps the fp16 P tile from overflowing, and scales back.
__device__ __forceinline__ float pow2_above(float m) {
    if (!(m > 0.f)) return 1.f;
    int e;
    frexpf(m, &e);  // m = f 2^e, 0.5 <= f < 1
    return ldexpf(1.f, e);
}

// x-gradient signal bound: guard[2] = the largest |b| (float bits), written by tc_bmax_kernel.
__global__ void __launch_bounds__(256) tc_bmax_kernel(const float *b, int64_t n, unsigned *gmax) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    float m = r < n ? fabsf(__ldg(b + r)) : 0.f;  // a NaN becomes NaN bits, above +inf: the guard fails
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = __uint_as_float(max(__float_as_uint(m), __float_as_uint(__shfl_xor_sync(0xffffffffu, m, o))));
    if ((threadIdx.x & 31) == 0) atomicMax(gmax, __float_as_uint(m));
}

// ---------------------------------------------------------------------------
// Operand prepass: row r of src (D floats) -> augmented, split fp16 row of 64.
// is_x: A = [2x', -|x'|^2, -1]; else B = [y', 1, |y'|^2].  Rows past `rows` are
// zero.  guard receives the largest |.'|^2 (as float bits; non-negative floats
// order like unsigned integers).  With b non-null, bpad[r] = b[r] (0 past `rows`).
// ---------------------------------------------------------------------------
// LogSumExp (lse): slot D + 2 is the weight slot, 1 in A; in B (fpad non-null, b the
// log-weights w) block k of 256 threads is tile k of the B operands, its frame
// F_k = max over the tile of w' = w log2 e goes to fpad[k] and the slot holds
// max(w'_r - F_k, -1024) <= 0 (-1024 past `rows`), so every term 2^(t + slot) of the
// tile is at most 1 in the frame F_k.
// bmax non-null (the x-gradient): bpad[r] = b[r] / 2^e in point order (the gradient's
// evaluation reads it so), 2^e = pow2_above(largest |b|), instead of the Sum's per-thread order.
__global__ void __launch_bounds__(256) tc_prep_kernel(const float *src, int64_t rows, int64_t rows_pad, int D,
                                                      float c, int is_x, int lse, __half *hi, __half *lo,
                                                      unsigned *guard, const float *b, float *bpad, float *fpad,
                                                      const unsigned *bmax, float *carry, int carry_w) {
    __shared__ float wmax[8];
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows_pad) return;  // with fpad, rows_pad is a multiple of 256: whole blocks leave together
    const bool live = r < rows;
    float wslot = is_x ? 1.f : 0.f;
    if (fpad) {
        const float wl = live ? 1.4426950408889634f * __ldg(b + r) : -__int_as_float(0x7f800000);
        float m = wl;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
        __syncthreads();
        float F = wmax[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) F = fmaxf(F, wmax[k]);
        if (F == -__int_as_float(0x7f800000)) F = 0.f;  // no weight in the tile: any frame
        wslot = (wl - F < -1024.f) ? -1024.f : wl - F;    // a NaN weight stays NaN
        if (threadIdx.x == 0) fpad[blockIdx.x] = F;
    }
    const float *row = src + (live ? r : 0) * D;
    float n = 0.f;
    if (live) {
        for (int d = 0; d < D; ++d) {
            const float s = c * __ldg(row + d);
            n = fmaf(s, s, n);
        }
        atomicMax(guard, __float_as_uint(n));
        if (carry)  // K-min: no list published for the row yet
            for (int k = 0; k < carry_w; ++k) carry[r * carry_w + k] = __int_as_float(0x7f800000);
    }
    if (bpad && !fpad && bmax) {
        const float m = __uint_as_float(*bmax);
        const float inv = (m <= 3.0e38f) ? 1.f / pow2_above(m) : 0.f;  // an exact power of two
        bpad[r] = live ? __ldg(b + r) * inv : 0.f;
    } else if (bpad && !fpad) {
        // Sum: b in the order the evaluation threads read it.  Column c of a 256-point tile
        // is c0 + 8 kk + 2 q + e (c0 = 0 or 128, kk < 16, q < 4, e < 2) and thread q of each
        // quad of lanes takes columns c0 + 8 kk + 2 q + e, so it goes to c0 + 32 q + 2 kk + e:
        // one thread's 32 values are contiguous.
        const int64_t c = r % kCols, hv = c / 128, cc = c % 128;
        const int64_t dst = (r - c) + 128 * hv + 32 * ((cc % 8) / 2) + 2 * (cc / 8) + (cc % 2);
        bpad[dst] = live ? __ldg(b + r) : 0.f;
    }
    const float scale = is_x ? 2.f * c : c;
    const float v_d = is_x ? -n : 1.f, v_d1 = is_x ? -1.f : n;
    uint4 *ph = reinterpret_cast<uint4 *>(hi + r * 64);
    uint4 *pl = lo ? reinterpret_cast<uint4 *>(lo + r * 64) : nullptr;  // null: the high halves only
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        __align__(16) __half h[8];
        __align__(16) __half l[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int k = 8 * q + e;
            float v = 0.f;
            if (live) v = k < D ? scale * __ldg(row + k) : (k == D ? v_d : (k == D + 1 ? v_d1 : 0.f));
            if (lse && k == D + 2) v = wslot;  // dead B rows too: -1024, a term of 0
            h[e] = __float2half_rn(v);
            l[e] = __float2half_rn(v - __half2float(h[e]));
        }
        ph[q] = *reinterpret_cast<const uint4 *>(h);
        if (lo) pl[q] = *reinterpret_cast<const uint4 *>(l);
    }
}

// ---------------------------------------------------------------------------
// Main kernel: grid (ceil(M/128), S); block (row block, split) reduces its 128 rows
// over the split's tiles of 256 points.
// ---------------------------------------------------------------------------
template <bool LSE>
__device__ __forceinline__ void tc_body(const TcParams &p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    // barriers: a_full, full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain
    __shared__ __align__(8) uint64_t bars[1 + 2 * kStages + 4 + 1];
    if (!norms_ok(p.guard)) return;  // the CUDA-core kernel does this call's work

    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t s_a_hi = smem_addr(smem), s_a_lo = s_a_hi + kATileBytes;
    const uint32_t s_stage0 = s_a_hi + 2 * kATileBytes;  // stage s: B hi at +s*kStageBytes, B lo after it
    const uint32_t b_a_full = smem_addr(&bars[0]);
    const uint32_t b_full0 = b_a_full + 8, b_empty0 = b_full0 + 8 * kStages;
    const uint32_t b_accf0 = b_empty0 + 8 * kStages, b_acce0 = b_accf0 + 16, b_drain = b_acce0 + 16;
    volatile int *abort = &abort_flag;

    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kRows;
    const int64_t j_begin = (int64_t)blockIdx.y * p.chunk;
    const int64_t j_end = min(p.N, j_begin + p.chunk);
    const int T = j_end > j_begin ? (int)((j_end - j_begin + kCols - 1) / kCols) : 0;

    if (w == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (t == 0) {
        abort_flag = 0;
        mbar_init(b_a_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(b_full0 + 8 * s, 1);   // the producer's expect_tx arrival
            mbar_init(b_empty0 + 8 * s, 1);  // the MMAs' commit
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(b_accf0 + 8 * k, 1);           // the MMAs' commit
            mbar_init(b_acce0 + 8 * k, kEvalWarps);  // the evaluation warps
        }
        mbar_init(b_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_slot;

    // running compensated sums: Sum, four rows a thread (hs[h], ls[h]); LSE, one row (hs[0], ls[0])
    float hs[4] = {0.f, 0.f, 0.f, 0.f}, ls[4] = {0.f, 0.f, 0.f, 0.f};
    float m = -__int_as_float(0x7f800000);  // LSE: the frame of (hs[0], ls[0]), base 2
    if (w == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0 && T > 0) {
            mbar_expect_tx(b_a_full, 2 * kATileBytes);
            tma_2d(s_a_hi, &p.tm_a_hi, 0, (int)row0, b_a_full);
            tma_2d(s_a_lo, &p.tm_a_lo, 0, (int)row0, b_a_full);
            int issued = 0;
            for (int i = 0; i < T; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(b_empty0 + 8 * s, ((i / kStages) - 1) & 1, abort, p.wait_ns)) break;
                const int j0 = (int)(j_begin + (int64_t)i * kCols);
                const uint32_t st = s_stage0 + s * kStageBytes, full = b_full0 + 8 * s;
                if (p.starve) continue;  // test hook: no B tile ever arrives, so the MMA issuer's wait runs out
                mbar_expect_tx(full, kStageBytes);
                tma_2d(st, &p.tm_b_hi, 0, j0, full);
                tma_2d(st + kBTileBytes, &p.tm_b_lo, 0, j0, full);
                issued = i + 1;
            }
            if (*abort) {  // let the copies in flight land before shared memory is released
                mbar_drain(b_a_full, 0, p.wait_ns);
                for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                    mbar_drain(b_full0 + 8 * (i % kStages), (i / kStages) & 1, p.wait_ns);
            }
        }
    } else if (w == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && T > 0 && mbar_wait(b_a_full, 0, abort, p.wait_ns)) {
            bool issued = false;
            for (int i = 0; i < T; ++i) {
                const int s = i % kStages, k = i & 1;
                if (!mbar_wait(b_full0 + 8 * s, (i / kStages) & 1, abort, p.wait_ns)) break;
                if (i >= 2 && !mbar_wait(b_acce0 + 8 * k, ((i >> 1) - 1) & 1, abort, p.wait_ns)) break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t acc = tmem + (uint32_t)(k * kCols);
                const uint32_t bh = s_stage0 + s * kStageBytes, bl = bh + kBTileBytes;
                // K = 16 per MMA: 32 bytes of each swizzled operand row
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(acc, desc_sw128(s_a_hi + 32 * kk), desc_sw128(bh + 32 * kk), kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(acc, desc_sw128(s_a_hi + 32 * kk), desc_sw128(bl + 32 * kk), 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(acc, desc_sw128(s_a_lo + 32 * kk), desc_sw128(bh + 32 * kk), 1);
                commit(b_empty0 + 8 * s);
                commit(b_accf0 + 8 * k);
                issued = true;
            }
            if (*abort && issued) {  // let the MMAs in flight finish before TMEM is released
                commit(b_drain);
                mbar_drain(b_drain, 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- evaluation warps 2..9 ----------------
        const int quarter = w & 3, c0 = kEvalCols * ((w - 2) >> 2);
        const uint32_t lanes = (uint32_t)(32 * quarter) << 16;
        for (int i = 0; i < T; ++i) {
            const int k = i & 1;
            // LSE: the tile's frame, loaded before the wait so its latency is hidden
            const float F = LSE ? __ldg(p.fpad + j_begin / kCols + i) : 0.f;
            if (!mbar_wait(b_accf0 + 8 * k, (i >> 1) & 1, abort, p.wait_ns)) break;
            asm volatile("tcgen05.fence::after_thread_sync;");
            if (LSE) {
                // one row per lane (32x32b), the accumulator holds t + w' - F: nothing else to read
                uint32_t r[kEvalCols];
                tmem_ld128(tmem + lanes + (uint32_t)(k * kCols + c0), r);  // one load, one wait
                asm volatile("tcgen05.wait::ld.sync.aligned;");
                asm volatile("tcgen05.fence::before_thread_sync;");
                __syncwarp();
                if (lane == 0) mbar_arrive(b_acce0 + 8 * k);  // the MMAs of tile i+2 may overwrite it
                float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
                for (int q = 0; q < kEvalCols; q += 4) {
                    p0 += ex2_approx(__uint_as_float(r[q + 0]));
                    p1 += ex2_approx(__uint_as_float(r[q + 1]));
                    p2 += ex2_approx(__uint_as_float(r[q + 2]));
                    p3 += ex2_approx(__uint_as_float(r[q + 3]));
                }
                const float pt = (p0 + p1) + (p2 + p3);
                if (!(pt == 0.f)) {  // fold the tile (frame F) into the running (m, hi, lo)
                    const float mn = fmaxf(m, F);
                    const float so = ex2_approx(m - mn), sn = ex2_approx(F - mn);
                    hs[0] *= so;
                    ls[0] *= so;
                    two_sum_add(hs[0], ls[0], pt * sn);
                    m = mn;
                }
            } else {
                // four rows per thread (two 16x256b loads): rows 32 quarter + t/4 + 8 h (+16 for
                // the second load), columns c0 + 8 kk + 2 (t%4) + e; so a thread needs b at only
                // its 32 columns
                uint32_t r0[64], r1[64];
                tmem_ld16x256_x16(tmem + lanes + (uint32_t)(k * kCols + c0), r0);
                tmem_ld16x256_x16(tmem + lanes + (16u << 16) + (uint32_t)(k * kCols + c0), r1);
                asm volatile("tcgen05.wait::ld.sync.aligned;");
                asm volatile("tcgen05.fence::before_thread_sync;");
                __syncwarp();
                if (lane == 0) mbar_arrive(b_acce0 + 8 * k);  // the MMAs of tile i+2 may overwrite it
                // b of this thread's 32 columns, stored contiguously by the prepass
                const float4 *bv =
                    reinterpret_cast<const float4 *>(p.bpad + j_begin + (int64_t)i * kCols + c0 + 32 * (lane & 3));
                float2 acc[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    float4 b4;
                    if ((kk & 1) == 0) b4 = __ldg(bv + kk / 2);
                    const float2 b2 = (kk & 1) ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 e0 = make_float2(ex2_approx(__uint_as_float(r0[4 * kk + 2 * h])),
                                                      ex2_approx(__uint_as_float(r0[4 * kk + 2 * h + 1])));
                        const float2 e1 = make_float2(ex2_approx(__uint_as_float(r1[4 * kk + 2 * h])),
                                                      ex2_approx(__uint_as_float(r1[4 * kk + 2 * h + 1])));
                        acc[h] = __ffma2_rn(e0, b2, acc[h]);
                        acc[2 + h] = __ffma2_rn(e1, b2, acc[2 + h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < 4; ++h) two_sum_add(hs[h], ls[h], acc[h].x + acc[h].y);
            }
        }
    }

    __syncthreads();
    const bool ok = !*abort;
    if (!ok && t == 0) atomicOr(&g_tc_status, 1u);
    float *red = reinterpret_cast<float *>(smem);
    if (!LSE && w >= 2) {
        // the four lanes t^1, t^2, t^3 hold the same rows: combine them in a fixed order
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1)
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float h2 = __shfl_xor_sync(0xffffffffu, hs[h], o), l2 = __shfl_xor_sync(0xffffffffu, ls[h], o);
                two_sum_add(hs[h], ls[h], h2);
                ls[h] += l2;
            }
    }
    // warps 6..9 hand their row sums (and LSE frames) to warps 2..5 through the idle A tile
    if (w >= 6) {
        if (LSE) {
            red[32 * (w & 3) + lane] = hs[0];
            red[kRows + 32 * (w & 3) + lane] = ls[0];
            red[2 * kRows + 32 * (w & 3) + lane] = m;
        } else if ((lane & 3) == 0) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int rl = 32 * (w & 3) + (lane >> 2) + 8 * h;
                red[rl] = hs[h];
                red[kRows + rl] = ls[h];
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (w == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));

    const float nan = __int_as_float(0x7fc00000);
    if (LSE && w >= 2 && w < 6) {
        const int rl = 32 * (w & 3) + lane;
        float hi = hs[0], lo = ls[0];
        float h2 = red[rl], l2 = red[kRows + rl];
        {  // bring both halves to the larger frame
            const float m2 = red[2 * kRows + rl], mn = fmaxf(m, m2);
            const float s1 = mn == -__int_as_float(0x7f800000) ? 0.f : ex2_approx(m - mn);
            const float s2 = mn == -__int_as_float(0x7f800000) ? 0.f : ex2_approx(m2 - mn);
            hi *= s1;
            lo *= s1;
            h2 *= s2;
            l2 *= s2;
            m = mn;
        }
        two_sum_add(hi, lo, h2);
        lo += l2;
        const int64_t i = row0 + rl;
        if (i < p.M) {
            const int64_t o = (int64_t)blockIdx.y * p.M + i;
            // the CUDA-core LogSumExp's output and partials: L = ln 2 (m + log2 tot); (m, tot)
            const float tot = hi + lo;
            const float ninf = -__int_as_float(0x7f800000);
            if (p.S == 1) {
                p.out[i] = !ok ? nan : tot > 0.f ? (float)(0.6931471805599453 * ((double)m + log2((double)tot))) : ninf;
            } else {
                p.ws0[o] = !ok ? nan : tot > 0.f ? m : ninf;
                p.ws1[o] = ok ? tot : 0.f;
            }
        }
    }
    if (!LSE && w >= 2 && w < 6 && (lane & 3) == 0) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int rl = 32 * (w & 3) + (lane >> 2) + 8 * h;
            float hi = hs[h], lo = ls[h];
            two_sum_add(hi, lo, red[rl]);
            lo += red[kRows + rl];
            const int64_t i = row0 + rl;
            if (i < p.M) {
                const int64_t o = (int64_t)blockIdx.y * p.M + i;
                if (p.S == 1) {
                    p.out[i] = ok ? hi + lo : nan;
                } else {
                    p.ws0[o] = ok ? hi : nan;
                    p.ws1[o] = ok ? lo : 0.f;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreadsTc, 1) tc_sum_kernel(const __grid_constant__ TcParams p) {
    tc_body<false>(p);
}
__global__ void __launch_bounds__(kThreadsTc, 1) tc_lse_kernel(const __grid_constant__ TcParams p) {
    tc_body<true>(p);
}

// One warp reads (writes) n consecutive 32-bit columns of its 32 TMEM lanes (one row per lane).
__device__ __forceinline__ void tmem_ld32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr), "r"(r[0]),"r"(r[1]),"r"(r[2]),"r"(r[3]),"r"(r[4]),"r"(r[5]),"r"(r[6]),"r"(r[7]),"r"(r[8]),"r"(r[9]),"r"(r[10]),"r"(r[11]),"r"(r[12]),"r"(r[13]),"r"(r[14]),"r"(r[15])
                 : "memory");
}

// ---------------------------------------------------------------------------
// K-min on the tensor cores (tc_knn_kernel), 32 <= D <= 62: a screen.  One product of the
// operands' high fp16 halves, A_hi . B_hi^T with A = [2x, -|x|^2, -1] and B = [y, 1, |y|^2]
// (prescale 1), gives S_ij = -|x_i - y_j|^2 up to
//   2^-8 (|x_i|^2 + max_j |y_j|^2) + 2^-24 (D + 2).
// The relative part: every operand is its fp16 half within 2^-11 of itself, so a product
// within 2^-10 (and a little) of itself, and the products' magnitudes sum to at most
// 2 (|x|^2 + |y|^2); the fp32 accumulation of 64 of them adds 2^-18 of that.  The absolute
// part: an operand below fp16's normal range (under 2^-14; the tensor cores keep fp16
// subnormals) is rounded to a multiple of 2^-24, within 2^-25, and meets the other
// operand's entries (sum over d of |y_d| + 2 |x_d| + 2 <= 1.5 D + |x|^2 + |y|^2 + 2).
// A point passes when -S_ij is at most T + margin, where T is the K-th distance of the row's
// list: this block's own, which starts from the best list any block of the row has shared
// (the row's shared list: distances only, in the workspace).  Its entries enter as stand-ins,
// which rank after any point of equal distance and are never reported.  Why no point of
// the row's final K fails the screen or is displaced: the shared lists hold distances of
// real points of other blocks, sorted, so slot k of one (even one read while another block
// rewrites it, slot by slot) is at least the k-th smallest distance of all the row's other
// points; hence slot k of this list is at least the k-th smallest of all the row's points,
// and a point of this split that the list turns away (or pushes past slot K - 1) has K
// points of the row ranking before it.  A block reads the shared list whole only at its
// start (so it never holds its own points), afterwards only its K-th slot as a bound, and
// writes its own list there after a tile where it became better than the shared one.
// Passing points get the direct fp32 distance (sum over d of (x_d - y_d)^2, in order) and
// enter the list when they rank before its K-th entry, in increasing j, so equal distances
// keep the lower index; the lists are the CUDA-core kernel's up to the rounding of the
// direct distance.  Chained this way, the splits of a row together take about the
// candidates of one list over all N points, K (1 + ln(N / K)), where lists that each started
// empty would take K ln(N_split / K) apiece.
// Block: 256 rows (two A tiles of 128, one MMA each, so that every B tile read from L2
// serves 256 rows) against tiles of 128 points; TMEM holds two tiles' products (two
// buffers of two 128-column accumulators).  Evaluation warp w owns rows 128 h + 32 q..
// (q = w mod 4, h = (w - 2) / 4): its TMEM lanes 32 q.. of accumulator h, one list a row.
// A chunk of 64 columns holding no pass costs one three-input max a column pair.  The
// operands are only the high halves: a B stage is 16 KB and ten of them are in flight.
// ---------------------------------------------------------------------------
constexpr int kKRows = kTcKnnRows;  // 2 x kRows
constexpr int kKCols = kTcKnnCols;
constexpr int kKBTileBytes = kKCols * 128;  // 128 points x 64 fp16
constexpr int kKStages = 10;
constexpr int kKChunk = 64;  // columns a TMEM load and a screen test
static_assert(kKRows == 2 * kRows, "two A tiles a block");
static_assert(2 * kATileBytes + kKStages * kKBTileBytes + 1024 <= kSmemBytes, "K-min stages within the Sum's shared memory");
static_assert(kKCols % kKChunk == 0 && 4 * kKCols <= kTmemCols, "whole chunks; two buffers of two accumulators");
static_assert(kEvalWarps == 8, "two warps a TMEM lane quarter");
// M = 128, N = kKCols, both K-major
constexpr uint32_t kIdescK = (1u << 4) | ((uint32_t)(kKCols >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);

__device__ __forceinline__ bool knn_norms_ok(const unsigned *guard) {
    return __uint_as_float(guard[0]) + __uint_as_float(guard[1]) <= kTcKnnNormLimit;
}

// Inserts (q, j) into a list sorted by (d, j) when it ranks above its last entry (unfilled
// slots are (+inf, -1)).
template <int KP>
__device__ __forceinline__ void knn_insert_dj(float (&dk)[KP], int (&ik)[KP], float q, int j) {
    // (q, j) ranks before (d, i): a smaller distance, or an equal one with a lower index; an
    // unfilled slot (+inf, -1) ranks after every real entry
    auto before = [](float q, int j, float d, int i) { return q < d || (q == d && j >= 0 && (i < 0 || j < i)); };
    // slot k takes the old slot k-1 when the new entry ranks before it, the new entry when it
    // lands exactly at k, and keeps its value otherwise (as knn_insert, with the index tie-break)
#pragma unroll
    for (int k = KP - 1; k > 0; --k) {
        const float da = dk[k - 1], db = dk[k];
        const int ia = ik[k - 1], ib = ik[k];
        const bool above = before(q, j, da, ia), here = before(q, j, db, ib);
        dk[k] = above ? da : (here ? q : db);
        ik[k] = above ? ia : (here ? j : ib);
    }
    if (before(q, j, dk[0], ik[0])) {
        dk[0] = q;
        ik[0] = j;
    }
}

// dk[K - 1] (ik[K - 1]) with constant indices only, 1 <= K <= KP.  Each slot passes through
// an empty asm so that the selects are not folded back into an indexed load, which would move
// the list from registers to local memory.
template <int KP>
__device__ __forceinline__ float knn_kth(const float (&dk)[KP], int K) {
    float v = dk[0];
#pragma unroll
    for (int k = 1; k < KP; ++k) {
        float c = dk[k];
        asm("" : "+f"(c));
        v = k == K - 1 ? c : v;
    }
    return v;
}
template <int KP>
__device__ __forceinline__ int knn_kth(const int (&ik)[KP], int K) {
    int v = ik[0];
#pragma unroll
    for (int k = 1; k < KP; ++k) {
        int c = ik[k];
        asm("" : "+r"(c));
        v = k == K - 1 ? c : v;
    }
    return v;
}

// Index of a stand-in entry: a distance taken from the row's shared list, which ranks after
// every point of equal distance and is never reported.
constexpr int kKnnStandIn = 0x7fffffff;

// Direct fp32 squared distance between row i of x and point j of y (D coordinates each),
// summed in coordinate order; G coordinates of each at a time are in flight.
template <int G>
__device__ __forceinline__ float tc_knn_dist(const float *xi, const float *yj, int D) {
    float q = 0.f;
    int d = 0;
    for (; d + G <= D; d += G) {
        float a[G], b[G];
#pragma unroll
        for (int e = 0; e < G; ++e) {
            a[e] = __ldg(xi + d + e);
            b[e] = __ldg(yj + d + e);
        }
#pragma unroll
        for (int e = 0; e < G; ++e) q = fmaf(a[e] - b[e], a[e] - b[e], q);
    }
    for (; d < D; ++d) {
        const float df = __ldg(xi + d) - __ldg(yj + d);
        q = fmaf(df, df, q);
    }
    return q;
}

// The columns c of r whose screened distance -r[c] is at most thr, as two 32-bit masks.
__device__ __forceinline__ void knn_pass_mask(const uint32_t (&r)[kKChunk], float thr, uint32_t &m0, uint32_t &m1) {
    m0 = 0u;
    m1 = 0u;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        m0 |= !(-__uint_as_float(r[c]) > thr) ? (1u << c) : 0u;
        m1 |= !(-__uint_as_float(r[32 + c]) > thr) ? (1u << c) : 0u;
    }
}

template <int KP>
__global__ void __launch_bounds__(kThreadsTc, 1) tc_knn_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    // barriers: a_full, full[kKStages], empty[kKStages], acc_full[2], acc_empty[2], drain
    __shared__ __align__(8) uint64_t bars[1 + 2 * kKStages + 4 + 1];
    if (!knn_norms_ok(p.guard)) return;  // the CUDA-core kernel does this call's work

    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t s_a = smem_addr(smem), s_stage0 = s_a + 2 * kATileBytes;
    const uint32_t b_a_full = smem_addr(&bars[0]);
    const uint32_t b_full0 = b_a_full + 8, b_empty0 = b_full0 + 8 * kKStages;
    const uint32_t b_accf0 = b_empty0 + 8 * kKStages, b_acce0 = b_accf0 + 16, b_drain = b_acce0 + 16;
    volatile int *abort = &abort_flag;

    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kKRows;
    const int64_t j_begin = (int64_t)blockIdx.y * p.chunk;
    const int64_t j_end = min(p.N, j_begin + p.chunk);
    const int T = j_end > j_begin ? (int)((j_end - j_begin + kKCols - 1) / kKCols) : 0;

    if (w == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (t == 0) {
        abort_flag = 0;
        mbar_init(b_a_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(b_full0 + 8 * s, 1);
            mbar_init(b_empty0 + 8 * s, 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(b_accf0 + 8 * k, 1);
            mbar_init(b_acce0 + 8 * k, kEvalWarps);
        }
        mbar_init(b_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_slot;

    // evaluation warps 2..9: row i (one a lane) and its list
    const int quarter = w & 3, h = (w - 2) >> 2;
    const int64_t i = row0 + kRows * h + 32 * quarter + lane;
    const bool live = w >= 2 && i < p.M;
    float dk[KP];
    int ik[KP];
#pragma unroll
    for (int k = 0; k < KP; ++k) {
        dk[k] = __int_as_float(0x7f800000);
        ik[k] = -1;
    }
    if (w == 0) {
        // ---------------- TMA producer: the high halves only ----------------
        if (lane == 0 && T > 0) {
            mbar_expect_tx(b_a_full, 2 * kATileBytes);
            tma_2d(s_a, &p.tm_a_hi, 0, (int)row0, b_a_full);
            tma_2d(s_a + kATileBytes, &p.tm_a_hi, 0, (int)(row0 + kRows), b_a_full);
            int issued = 0;
            for (int n = 0; n < T; ++n) {
                const int s = n % kKStages;
                if (n >= kKStages && !mbar_wait(b_empty0 + 8 * s, ((n / kKStages) - 1) & 1, abort, p.wait_ns)) break;
                const int j0 = (int)(j_begin + (int64_t)n * kKCols);
                const uint32_t full = b_full0 + 8 * s;
                if (p.starve) continue;  // test hook: no B tile ever arrives, so the MMA issuer's wait runs out
                mbar_expect_tx(full, kKBTileBytes);
                tma_2d(s_stage0 + s * kKBTileBytes, &p.tm_b_hi, 0, j0, full);
                issued = n + 1;
            }
            if (*abort) {
                mbar_drain(b_a_full, 0, p.wait_ns);
                for (int n = issued > kKStages ? issued - kKStages : 0; n < issued; ++n)
                    mbar_drain(b_full0 + 8 * (n % kKStages), (n / kKStages) & 1, p.wait_ns);
            }
        }
    } else if (w == 1) {
        // ---------------- MMA issuer: S_h = A_h . B^T (h = 0, 1), four K steps of 16 each ----
        if (lane == 0 && T > 0 && mbar_wait(b_a_full, 0, abort, p.wait_ns)) {
            bool issued = false;
            for (int n = 0; n < T; ++n) {
                const int s = n % kKStages, k = n & 1;
                if (!mbar_wait(b_full0 + 8 * s, (n / kKStages) & 1, abort, p.wait_ns)) break;
                if (n >= 2 && !mbar_wait(b_acce0 + 8 * k, ((n >> 1) - 1) & 1, abort, p.wait_ns)) break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t bh = s_stage0 + s * kKBTileBytes;
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const uint32_t acc = tmem + (uint32_t)((2 * k + a) * kKCols);
                    const uint32_t ah = s_a + (uint32_t)(a * kATileBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16(acc, desc_sw128(ah + 32 * kk), desc_sw128(bh + 32 * kk), kk > 0, kIdescK);
                }
                commit(b_empty0 + 8 * s);
                commit(b_accf0 + 8 * k);
                issued = true;
            }
            if (*abort && issued) {
                commit(b_drain);
                mbar_drain(b_drain, 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- evaluation warps 2..9: one row a lane, one list a row ----------------
        const uint32_t lanes = (uint32_t)(32 * quarter) << 16;
        const float *xi = p.x + (live ? i : 0) * p.D;
        float *const cl = p.carry + (live ? i : 0) * KP;  // the row's shared list
        // this row's |x|^2 (fp32) and the screen's margin
        float nx = 0.f;
        for (int d = 0; d < p.D; ++d) nx = fmaf(__ldg(xi + d), __ldg(xi + d), nx);
        const float margin = 0x1p-8f * (nx + __uint_as_float(p.guard[1])) + 0x1p-24f * (float)(p.D + 2);
        const float inf = __int_as_float(0x7f800000);
        // the list starts from the row's shared one: its distances enter as stand-ins (index
        // kKnnStandIn), which rank after every point of equal distance and are never reported
        if (live) {
#pragma unroll
            for (int k = 0; k < KP; ++k) {
                const float v = __ldcg(cl + k);
                if (v < inf) knn_insert_dj<KP>(dk, ik, v, kKnnStandIn);
            }
        }
        float kth = knn_kth<KP>(dk, p.K);  // this list's K-th distance
        float pub = kth;                    // the K-th it last published (or started from)
        float thr = kth + margin;           // -S must be at most this to pass
        for (int it = 0; it < T; ++it) {
            const int k = it & 1;
            // the row's shared K-th (read before the wait: it is in flight meanwhile)
            const float gth = live ? __ldcg(cl + (p.K - 1)) : inf;
            // (the warp leaves together)
            if (!__all_sync(0xffffffffu, mbar_wait(b_accf0 + 8 * k, (it >> 1) & 1, abort, p.wait_ns))) break;
            asm volatile("tcgen05.fence::after_thread_sync;");
            const int64_t jt = j_begin + (int64_t)it * kKCols;
#pragma unroll 1
            for (int ch = 0; ch < kKCols / kKChunk; ++ch) {
                uint32_t r[kKChunk];
                tmem_ld32x32b_x64(tmem + lanes + (uint32_t)((2 * k + h) * kKCols + kKChunk * ch), r);
                asm volatile("tcgen05.wait::ld.sync.aligned;");
                // the chunk's largest S (nearest point): one test for 64 columns
                float mx = __uint_as_float(r[0]);
#pragma unroll
                for (int c = 1; c < kKChunk - 1; c += 2) mx = fmax3(mx, __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
                mx = fmaxf(mx, __uint_as_float(r[kKChunk - 1]));
                if (live && !(-mx > thr)) {
                    // the passing columns, walked in increasing j; after an insertion the
                    // threshold falls and the columns still to come are screened again
                    uint32_t m0, m1;
                    knn_pass_mask(r, thr, m0, m1);
                    while (m0 | m1) {
                        const int c = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
                        if (m0) m0 &= m0 - 1; else m1 &= m1 - 1;
                        const int64_t j = jt + kKChunk * ch + c;
                        if (j >= j_end) break;  // the rest of the chunk is past the split too
                        // (longer lists leave fewer registers for the loads in flight)
                        const float q = tc_knn_dist<KP <= 16 ? 16 : 8>(xi, p.y + j * p.D, p.D);
                        // (q, j) enters when it ranks before the K-th entry: a smaller distance,
                        // or an equal one held by a stand-in (the list's own points have lower j)
                        if (q < kth || (q == kth && knn_kth<KP>(ik, p.K) == kKnnStandIn)) {
                            knn_insert_dj<KP>(dk, ik, q, (int)j);
                            kth = knn_kth<KP>(dk, p.K);
                            thr = fminf(kth, gth) + margin;
                            uint32_t n0, n1;
                            knn_pass_mask(r, thr, n0, n1);
                            m0 &= n0;
                            m1 &= n1;
                        }
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;");
            __syncwarp();
            if (lane == 0) mbar_arrive(b_acce0 + 8 * k);  // the MMAs of tile it+2 may overwrite it
            if (live && kth < pub && kth < gth) {  // a better list than the row's: share it
#pragma unroll
                for (int e = 0; e < KP; ++e) __stcg(cl + e, dk[e]);
                pub = kth;
            }
            thr = fminf(kth, gth) + margin;
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    const bool ok = !*abort;
    if (!ok && t == 0) atomicOr(&g_tc_status, 1u);
    if (w == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    if (live) {
        // the list's own points in order (the stand-ins left out), then empty slots
        const float nan = __int_as_float(0x7fc00000), inf = __int_as_float(0x7f800000);
        const int width = p.S == 1 ? p.K : KP;
        const int64_t o = p.S == 1 ? i * p.K : ((int64_t)blockIdx.y * p.M + i) * KP;
        int32_t *const oi = (p.S == 1 ? p.idx : p.wsi) + o;
        float *const od = p.S == 1 ? (p.out ? p.out + o : nullptr) : p.ws0 + o;  // (the distances may be left out)
        int n = 0;
#pragma unroll
        for (int k = 0; k < KP; ++k) {
            if (k >= p.K || ik[k] < 0 || ik[k] == kKnnStandIn) continue;
            oi[n] = ok ? ik[k] : -1;
            if (od) od[n] = ok ? dk[k] : nan;
            ++n;
        }
        for (; n < width; ++n) {
            oi[n] = -1;
            if (od) od[n] = ok ? inf : nan;
        }
    }
}

// ---------------------------------------------------------------------------
// x-gradient (tc_grad_kernel), 32 <= D <= 62, E = 1:
//   gx_id = gscale g_i sum_j k_ij b_j (x'_id - y'_jd) = gscale g_i (x'_id s0_i - s_id),
//   s0_i = sum_j P_ij,  s_id = sum_j P_ij y'_jd,  P_ij = k_ij b_j = 2^(S_ij) b_j.
// Both contractions run on the tensor cores.  Per tile of kGCols = 128 points:
//   MMA 1: S = A . B^T as for the Sum (N = 128), into one of two TMEM accumulators;
//   evaluation warps: P = 2^S b in fp32, split P = hi + lo (fp16 each) and written into
//     the shared-memory P tile (K-major over the tile's points, 128-byte swizzle);
//   MMA 2: D2 += P . [y' | 1 | ...], where the right operand is the same B tile read
//     MN-major (its point rows are now the K dimension): column d < D of D2 is s_id and
//     column D (B's slot of 1) is s0_i; products Phi.Bhi + Phi.Blo + Plo.Bhi, fp32, in one
//     of two further TMEM accumulators, each summing kGGroup tiles;
//   evaluation warps fold each group's D2 into compensated (TwoSum) running sums, kept in
//     TMEM too, so that a warp's registers hold only the tile in flight.
// s0 and s come from the same rounded P, so the cancellation in x' s0 - s leaves only the
// operands' own rounding (about 2^-22 of them) against sum_j |P_ij| |x'_id - y'_jd|, the
// tolerance's scale.  The MMA issuer runs the first products two tiles ahead of the
// second, so the next S is computed while the warps turn the last one into P.  A tile's B
// stage is released only by its second product, two tiles after its first: of the four
// stages, the one beyond those three is the TMA's lookahead.
// Block = 18 warps (TMA producer, MMA issuer, 16 evaluation warps: the evaluation is
// latency-bound, so four warps a scheduler, at 96 registers each); TMEM columns [0, 256):
// two S accumulators of 128; [256, 384): two D2 accumulators of 64; [384, 512): the
// running sums (hi at 384 + c, lo at 448 + c for D2 column c).  Evaluation warp w reads
// TMEM lanes 32 (w mod 4).. (its rows) and takes S columns 32 q.. and D2 columns 16 q..
// (q = (w - 2) / 4).
// ---------------------------------------------------------------------------
constexpr int kGCols = kTcGradCols;
constexpr int kGStages = 4;  // the second product holds a tile's B stage two tiles longer
constexpr int kGEvalWarps = 16;                 // four per TMEM lane quarter: 32 S columns each
constexpr int kGThreads = kTcGradThreads;
static_assert(kGThreads == 64 + 32 * kGEvalWarps, "warp roles");
constexpr int kGGroup = 4;                      // tiles summed in one D2 accumulator
constexpr int kGBTileBytes = kGCols * 128;      // 128 points x 64 fp16
constexpr int kGStageBytes = 2 * kGBTileBytes;  // hi, lo
constexpr int kGPHalfBytes = kRows * 128;       // 128 rows x 64 points fp16: one K half of P
constexpr int kGPBytes = 4 * kGPHalfBytes;      // hi (two K halves), lo (two K halves)
constexpr int kGSmemBytes = 2 * kATileBytes + kGStages * kGStageBytes + kGPBytes + 1024;
static_assert(kGSmemBytes + 1024 <= 227 * 1024, "shared memory per block (the static part is under 1 KB)");
static_assert(kGPBytes >= kRows * 64 * 2 * 4, "the P tile holds the final (hi, lo) sums");
// MMA 1: M = 128, N = 128, both K-major.  MMA 2: M = 128, N = 64, A K-major, B MN-major.
constexpr uint32_t kIdescG1 = (1u << 4) | ((uint32_t)(kGCols >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
constexpr uint32_t kIdescG2 = (1u << 4) | (1u << 16) | ((uint32_t)(64 >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
constexpr int kGTmemS = 0, kGTmemD2 = 2 * kGCols, kGTmemRun = kGTmemD2 + 128;

__global__ void __launch_bounds__(kGThreads, 1) tc_grad_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    // a_full, full[4], empty[4], s_full[2], s_empty[2], d2_full[2], d2_empty[2], p_full, p_empty, drain
    __shared__ __align__(8) uint64_t bars[1 + 2 * kGStages + 8 + 3];
    __shared__ unsigned pmx[kRows];  // largest |P| of each row (float bits: non-negative, so ordered as integers)
    if (!norms_ok(p.guard) || !(__uint_as_float(p.guard[2]) <= 3.0e38f))
        return;  // the CUDA-core kernel does this call's work

    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t s_a_hi = smem_addr(smem), s_a_lo = s_a_hi + kATileBytes;
    const uint32_t s_stage0 = s_a_hi + 2 * kATileBytes;
    uint8_t *const pbuf = smem + 2 * kATileBytes + kGStages * kGStageBytes;
    const uint32_t s_p = smem_addr(pbuf);  // P hi: K halves at +0, +kGPHalfBytes; P lo after them
    const uint32_t b_a_full = smem_addr(&bars[0]);
    const uint32_t b_full0 = b_a_full + 8, b_empty0 = b_full0 + 8 * kGStages;
    const uint32_t b_sf0 = b_empty0 + 8 * kGStages, b_se0 = b_sf0 + 16;
    const uint32_t b_df0 = b_se0 + 16, b_de0 = b_df0 + 16;
    const uint32_t b_pfull = b_de0 + 16, b_pempty = b_pfull + 8, b_drain = b_pempty + 8;
    volatile int *abort = &abort_flag;

    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kRows;
    const int64_t j_begin = (int64_t)blockIdx.y * p.chunk;
    const int64_t j_end = min(p.N, j_begin + p.chunk);
    const int T = j_end > j_begin ? (int)((j_end - j_begin + kGCols - 1) / kGCols) : 0;

    if (w == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (t < kRows) pmx[t] = 0u;
    if (t == 0) {
        abort_flag = 0;
        mbar_init(b_a_full, 1);
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(b_full0 + 8 * s, 1);   // the producer's expect_tx arrival
            mbar_init(b_empty0 + 8 * s, 1);  // the second product's commit
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(b_sf0 + 8 * k, 1);           // first product's commit
            mbar_init(b_se0 + 8 * k, kGEvalWarps);  // S read by the evaluation warps
            mbar_init(b_df0 + 8 * k, 1);           // a group's last second product
            mbar_init(b_de0 + 8 * k, kGEvalWarps);  // D2 read by the evaluation warps
        }
        mbar_init(b_pfull, kGEvalWarps);           // P tile written
        mbar_init(b_pempty, 1);                    // P tile read by the second product
        mbar_init(b_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_slot;
    // evaluation warp w: TMEM lanes 32 (w mod 4).. (its rows), column part (w - 2) / 4: S columns
    // 32 part.., D2 columns 16 part..
    const int quarter = w & 3, part = (w - 2) >> 2, row_l = 32 * quarter + lane;
    const uint32_t lanes = (uint32_t)(32 * quarter) << 16;
    const uint32_t t_hi = tmem + lanes + (uint32_t)(kGTmemRun + 16 * part);  // this warp's running sums
    const uint32_t t_lo = t_hi + 64;

    if (w == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0 && T > 0) {
            mbar_expect_tx(b_a_full, 2 * kATileBytes);
            tma_2d(s_a_hi, &p.tm_a_hi, 0, (int)row0, b_a_full);
            tma_2d(s_a_lo, &p.tm_a_lo, 0, (int)row0, b_a_full);
            int issued = 0;
            for (int i = 0; i < T; ++i) {
                const int s = i % kGStages;
                if (i >= kGStages && !mbar_wait(b_empty0 + 8 * s, ((i / kGStages) - 1) & 1, abort, p.wait_ns)) break;
                const int j0 = (int)(j_begin + (int64_t)i * kGCols);
                const uint32_t st = s_stage0 + s * kGStageBytes, full = b_full0 + 8 * s;
                if (p.starve) continue;  // test hook: no B tile ever arrives, so the MMA issuer's wait runs out
                mbar_expect_tx(full, kGStageBytes);
                tma_2d(st, &p.tm_b_hi, 0, j0, full);
                tma_2d(st + kGBTileBytes, &p.tm_b_lo, 0, j0, full);
                issued = i + 1;
            }
            if (*abort) {  // let the copies in flight land before shared memory is released
                mbar_drain(b_a_full, 0, p.wait_ns);
                for (int i = issued > kGStages ? issued - kGStages : 0; i < issued; ++i)
                    mbar_drain(b_full0 + 8 * (i % kGStages), (i / kGStages) & 1, p.wait_ns);
            }
        }
    } else if (w == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && T > 0 && mbar_wait(b_a_full, 0, abort, p.wait_ns)) {
            bool issued = false;
            // base descriptors: A (hi, lo after it), the B stages K-major and MN-major, P
            const uint64_t d_a = desc_sw128(s_a_hi), d_b = desc_sw128(s_stage0), d_bmn = desc_sw128_mn(s_stage0);
            const uint64_t d_p = desc_sw128(s_p);
            // second product of tile j: D2[group] += P(j) . B(j) (B read MN-major); then the P
            // tile and B(j)'s stage are free, and after a group's last tile its D2 is complete
            auto mma2 = [&](int j) -> bool {
                const int s = j % kGStages, g = j / kGGroup, kk = g & 1;
                const bool first = j % kGGroup == 0, last = j % kGGroup == kGGroup - 1 || j == T - 1;
                if (!mbar_wait(b_pfull, j & 1, abort, p.wait_ns)) return false;
                if (first && g >= 2 && !mbar_wait(b_de0 + 8 * kk, ((g >> 1) - 1) & 1, abort, p.wait_ns)) return false;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t acc = tmem + (uint32_t)(kGTmemD2 + kk * 64);
                const uint32_t so = (uint32_t)(s * kGStageBytes);
#pragma unroll
                for (int q = 0; q < kGCols / 16; ++q) {  // K = 16 points per product
                    const uint32_t pa = (uint32_t)((q >> 2) * kGPHalfBytes + 32 * (q & 3));
                    const uint32_t bb = so + (uint32_t)(16 * 128 * q);
                    const uint64_t dph = desc_add(d_p, pa), dpl = desc_add(d_p, pa + 2 * kGPHalfBytes);
                    const uint64_t dbh = desc_add(d_bmn, bb), dbl = desc_add(d_bmn, bb + kGBTileBytes);
                    mma_f16(acc, dph, dbh, (first && q == 0) ? 0u : 1u, kIdescG2);
                    mma_f16(acc, dph, dbl, 1, kIdescG2);
                    mma_f16(acc, dpl, dbh, 1, kIdescG2);
                }
                commit(b_pempty);
                commit(b_empty0 + 8 * s);
                if (last) commit(b_df0 + 8 * kk);
                return true;
            };
            bool ok = true;
            for (int i = 0; i < T && ok; ++i) {
                const int s = i % kGStages, k = i & 1;
                if (!mbar_wait(b_full0 + 8 * s, (i / kGStages) & 1, abort, p.wait_ns)) break;
                if (i >= 2 && !mbar_wait(b_se0 + 8 * k, ((i >> 1) - 1) & 1, abort, p.wait_ns)) break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t acc = tmem + (uint32_t)(kGTmemS + k * kGCols);
                const uint32_t so = (uint32_t)(s * kGStageBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(acc, desc_add(d_a, 32 * kk), desc_add(d_b, so + 32 * kk), kk > 0, kIdescG1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(acc, desc_add(d_a, 32 * kk), desc_add(d_b, so + kGBTileBytes + 32 * kk), 1, kIdescG1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(acc, desc_add(d_a, kATileBytes + 32 * kk), desc_add(d_b, so + 32 * kk), 1, kIdescG1);
                commit(b_sf0 + 8 * k);
                issued = true;
                if (i >= 2) ok = mma2(i - 2);  // the second products run two tiles behind
            }
            for (int j = T >= 2 ? T - 2 : 0; j < T && ok && !*abort; ++j) ok = mma2(j);
            if (*abort && issued) {  // let the products in flight finish before TMEM is released
                commit(b_drain);
                mbar_drain(b_drain, 0, p.wait_ns);
            }
        }
    } else {
        // ---------------- evaluation warps 2..17 ----------------
        // this row's P hi and lo in K half part / 2, 16-byte chunks 4 (part mod 2).. of the row
        uint8_t *const hb = pbuf + (part >> 1) * kGPHalfBytes + row_l * 128;
        uint8_t *const lb = pbuf + (2 + (part >> 1)) * kGPHalfBytes + row_l * 128;
        const int c0 = 4 * (part & 1), sw = row_l & 7;  // first chunk; 128-byte swizzle of the row
        {  // the running sums start at zero
            uint32_t z[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) z[c] = 0u;
            tmem_st32x32b_x16(t_hi, z);
            tmem_st32x32b_x16(t_lo, z);
            asm volatile("tcgen05.wait::st.sync.aligned;");
        }
        // group g's D2 (complete once its last second product is): fold into the running sums
        auto fold = [&](int g) -> bool {
            const int kk = g & 1;
            if (!mbar_wait(b_df0 + 8 * kk, (g >> 1) & 1, abort, p.wait_ns)) return false;
            asm volatile("tcgen05.fence::after_thread_sync;");
#pragma unroll
            for (int half = 0; half < 2; ++half) {  // 8 columns at a time (registers)
                uint32_t d[8], h[8], l[8];
                tmem_ld32x32b_x8(tmem + lanes + (uint32_t)(kGTmemD2 + kk * 64 + 16 * part + 8 * half), d);
                tmem_ld32x32b_x8(t_hi + 8 * half, h);
                tmem_ld32x32b_x8(t_lo + 8 * half, l);
                asm volatile("tcgen05.wait::ld.sync.aligned;");
                if (half == 1) {
                    asm volatile("tcgen05.fence::before_thread_sync;");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_de0 + 8 * kk);  // the second products of group g+2 may overwrite it
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float hv = __uint_as_float(h[c]), lv = __uint_as_float(l[c]);
                    two_sum_add(hv, lv, __uint_as_float(d[c]));
                    h[c] = __float_as_uint(hv);
                    l[c] = __float_as_uint(lv);
                }
                tmem_st32x32b_x8(t_hi + 8 * half, h);
                tmem_st32x32b_x8(t_lo + 8 * half, l);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;");
            return true;
        };
        bool ok = true;
        float pm = 0.f;  // largest |P| of this row's columns in this split
        // this warp's 32 signal values of the next tile, loaded a tile ahead (their latency
        // overlaps the P stores, the fold and the wait for S instead of following S)
        float4 bn[8];
        {
            const float4 *bv = reinterpret_cast<const float4 *>(p.bpad + j_begin + 32 * part);
#pragma unroll
            for (int q = 0; q < 8; ++q) bn[q] = T > 0 ? __ldg(bv + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int i = 0; i < T && ok; ++i) {
            const int k = i & 1;
            if (!mbar_wait(b_sf0 + 8 * k, (i >> 1) & 1, abort, p.wait_ns)) break;
            asm volatile("tcgen05.fence::after_thread_sync;");
            // P = 2^S b for this warp's 32 points, split into fp16 hi + lo, packed two points a
            // register: all of it before waiting for the P tile, which the second product of the
            // previous tile may still be reading
            uint32_t ph[16], pl[16];
            {
                uint32_t r[32];
                tmem_ld32x32b_x32(tmem + lanes + (uint32_t)(kGTmemS + k * kGCols + 32 * part), r);
                asm volatile("tcgen05.wait::ld.sync.aligned;");
                asm volatile("tcgen05.fence::before_thread_sync;");
                __syncwarp();
                if (lane == 0) mbar_arrive(b_se0 + 8 * k);  // the first product of tile i+2 may overwrite it
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    // two points an instruction (f32x2) for the products and the residuals
                    const float4 b4 = bn[q];
                    const float2 p01 = __fmul2_rn(make_float2(ex2_approx(__uint_as_float(r[4 * q + 0])),
                                                              ex2_approx(__uint_as_float(r[4 * q + 1]))),
                                                  make_float2(b4.x, b4.y));
                    const float2 p23 = __fmul2_rn(make_float2(ex2_approx(__uint_as_float(r[4 * q + 2])),
                                                              ex2_approx(__uint_as_float(r[4 * q + 3]))),
                                                  make_float2(b4.z, b4.w));
                    pm = fmax3(pm, fabsf(p01.x), fabsf(p01.y));
                    pm = fmax3(pm, fabsf(p23.x), fabsf(p23.y));
                    const __half2 h01 = __floats2half2_rn(p01.x, p01.y), h23 = __floats2half2_rn(p23.x, p23.y);
                    const float2 m1 = make_float2(-1.f, -1.f);
                    const float2 d01 = __ffma2_rn(__half22float2(h01), m1, p01);  // p - hi, exact
                    const float2 d23 = __ffma2_rn(__half22float2(h23), m1, p23);
                    const __half2 l01 = __floats2half2_rn(d01.x, d01.y);
                    const __half2 l23 = __floats2half2_rn(d23.x, d23.y);
                    ph[2 * q] = *reinterpret_cast<const uint32_t *>(&h01);
                    ph[2 * q + 1] = *reinterpret_cast<const uint32_t *>(&h23);
                    pl[2 * q] = *reinterpret_cast<const uint32_t *>(&l01);
                    pl[2 * q + 1] = *reinterpret_cast<const uint32_t *>(&l23);
                }
            }
            if (i + 1 < T) {
                const float4 *bv = reinterpret_cast<const float4 *>(p.bpad + j_begin + (int64_t)(i + 1) * kGCols + 32 * part);
#pragma unroll
                for (int q = 0; q < 8; ++q) bn[q] = __ldg(bv + q);
            }
            if (i >= 1 && !mbar_wait(b_pempty, (i - 1) & 1, abort, p.wait_ns)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {  // chunk c0 + cc = points 8 (c0 + cc).. of the K half, swizzled
                const int c = c0 + cc;
                *reinterpret_cast<uint4 *>(hb + ((c ^ sw) << 4)) = make_uint4(ph[4 * cc], ph[4 * cc + 1], ph[4 * cc + 2], ph[4 * cc + 3]);
                *reinterpret_cast<uint4 *>(lb + ((c ^ sw) << 4)) = make_uint4(pl[4 * cc], pl[4 * cc + 1], pl[4 * cc + 2], pl[4 * cc + 3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(b_pfull);
            if (i >= 1 && (i - 1) % kGGroup == kGGroup - 1) ok = fold((i - 1) / kGGroup);
        }
        if (ok && !*abort && T > 0) fold((T - 1) / kGGroup);
        atomicMax(&pmx[row_l], __float_as_uint(pm));
    }

    __syncthreads();
    const bool ok = !*abort;
    if (!ok && t == 0) atomicOr(&g_tc_status, 1u);
    // every row's 64 running sums (hi, lo) through the idle P tile, so every part sees s0 (column D)
    float *red = reinterpret_cast<float *>(pbuf);
    float ah[16], al[16];
    if (w >= 2) {
        uint32_t h[16], l[16];
        asm volatile("tcgen05.fence::after_thread_sync;");
        tmem_ld32x32b_x16(t_hi, h);
        tmem_ld32x32b_x16(t_lo, l);
        asm volatile("tcgen05.wait::ld.sync.aligned;");
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            ah[c] = __uint_as_float(h[c]);
            al[c] = __uint_as_float(l[c]);
            red[row_l * 64 + 16 * part + c] = ah[c];
            red[kRows * 64 + row_l * 64 + 16 * part + c] = al[c];
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (w == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
    if (w >= 2) {
        const int64_t i = row0 + row_l;
        // A row whose largest |P| in this split is below 2^-8 (every point far from it, or a small
        // signal there) keeps too few bits in the fp16 P tile: the CUDA-core kernel launched
        // after this one redoes this split's part of it (the flag says so), exactly.
        const bool weak = ok && T > 0 &&
                          __uint_as_float(pmx[row_l]) < 0x1p-8f;
        if (i < p.M && part == 0) p.flags[(int64_t)blockIdx.y * p.M + i] = weak ? 1 : 0;
        if (i < p.M && !weak) {
            const double s0 = (double)red[row_l * 64 + p.D] + (double)red[kRows * 64 + row_l * 64 + p.D];
            // the signal went in as b / 2^e (pow2_above of its largest magnitude): scale back
            const double sc =
                (double)p.gscale * (double)__ldg(p.g + i) * (double)pow2_above(__uint_as_float(p.guard[2]));
            const float nan = __int_as_float(0x7fc00000);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int d = 16 * part + c;
                if (d >= p.D) continue;
                const double xd = (double)(p.c * __ldg(p.x + i * p.D + d));
                const double v = (xd * s0 - ((double)ah[c] + (double)al[c])) * sc;
                const int64_t o = i * p.D + d;
                if (p.S == 1) {
                    p.out[o] = ok ? (float)v : nan;
                } else {
                    const int64_t wo = (int64_t)blockIdx.y * p.M * p.D + o;
                    const float hi = (float)v;
                    p.ws0[wo] = ok ? hi : nan;
                    p.ws1[wo] = ok ? (float)(v - (double)hi) : 0.f;
                }
            }
        }
    }
}

// Host: cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)f;
    });
    return fn;
}

// Tensor map over rows x 64 fp16 (128-byte rows), boxes of 64 x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap *m, const __half *base, int64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void *)base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tc_smem_bytes() { return kSmemBytes; }

// Opt both tensor-core kernels in to kSmemBytes of dynamic shared memory, once per device.
cudaError_t tc_set_attributes() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(tc_sum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmemBytes);
    for (const void *f : {(const void *)tc_knn_kernel<1>, (const void *)tc_knn_kernel<4>, (const void *)tc_knn_kernel<10>,
                          (const void *)tc_knn_kernel<16>, (const void *)tc_knn_kernel<32>})
        if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

cudaError_t tc_launch_bmax(const float *b, int64_t n, unsigned *guard, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    tc_bmax_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(b, n, guard + 2);
    return cudaGetLastError();
}

cudaError_t tc_launch_prep(const float *src, int64_t rows, int64_t rows_pad, int D, float c, bool is_x, bool lse,
                           __half *hi, __half *lo, unsigned *guard, const float *b, float *bpad, float *fpad,
                           cudaStream_t s, bool natural_b, float *carry, int carry_w) {
    // LSE frames: a prep block of 256 threads is one whole tile of kTcCols = 256 points
    if (fpad && rows_pad % 256) return cudaErrorInvalidValue;
    if (lse && (D + 2 >= 64 || (!is_x && !fpad))) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((rows_pad + 255) / 256);
    // the y side's guard slot is guard[1] of the call's guard words; the largest |b| is guard[2]
    tc_prep_kernel<<<blocks, 256, 0, s>>>(src, rows, rows_pad, D, c, is_x ? 1 : 0, lse ? 1 : 0, hi, lo, guard, b,
                                          bpad, fpad, natural_b ? guard + 1 : nullptr, carry, carry_w);
    return cudaGetLastError();
}

cudaError_t tc_launch_sum(const TcArgs &a, dim3 grid, cudaStream_t s) {
    TcParams p;
    if (a.m_pad % kRows || a.n_pad % kCols || a.chunk % kCols) return cudaErrorInvalidValue;
    if (!make_map(&p.tm_a_hi, a.a_hi, a.m_pad, kRows) || !make_map(&p.tm_a_lo, a.a_lo, a.m_pad, kRows) ||
        !make_map(&p.tm_b_hi, a.b_hi, a.n_pad, kCols) || !make_map(&p.tm_b_lo, a.b_lo, a.n_pad, kCols))
        return cudaErrorInvalidValue;
    p.bpad = a.bpad;
    p.fpad = a.fpad;
    p.out = a.out;
    p.ws0 = a.ws0;
    p.ws1 = a.ws1;
    p.guard = a.guard;
    p.wait_ns = a.wait_ns;
    p.starve = a.starve ? 1 : 0;
    p.M = a.M;
    p.N = a.N;
    p.chunk = a.chunk;
    p.S = a.S;
    cudaError_t e = tc_set_attributes();
    if (e != cudaSuccess) return e;
    if (a.lse)
        tc_lse_kernel<<<grid, kThreadsTc, kSmemBytes, s>>>(p);
    else
        tc_sum_kernel<<<grid, kThreadsTc, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

cudaError_t tc_launch_grad(const TcArgs &a, dim3 grid, cudaStream_t s) {
    TcParams p;
    if (a.m_pad % kRows || a.n_pad % kGCols || a.chunk % kGCols || a.D < 32 || a.D > 62) return cudaErrorInvalidValue;
    if (!make_map(&p.tm_a_hi, a.a_hi, a.m_pad, kRows) || !make_map(&p.tm_a_lo, a.a_lo, a.m_pad, kRows) ||
        !make_map(&p.tm_b_hi, a.b_hi, a.n_pad, kGCols) || !make_map(&p.tm_b_lo, a.b_lo, a.n_pad, kGCols))
        return cudaErrorInvalidValue;
    p.bpad = a.bpad;
    p.fpad = nullptr;
    p.out = a.out;
    p.ws0 = a.ws0;
    p.ws1 = a.ws1;
    p.guard = a.guard;
    p.wait_ns = a.wait_ns;
    p.starve = a.starve ? 1 : 0;
    p.M = a.M;
    p.N = a.N;
    p.chunk = a.chunk;
    p.S = a.S;
    p.x = a.x;
    p.g = a.g;
    p.D = a.D;
    p.c = a.c;
    p.gscale = a.gscale;
    p.flags = a.flags;
    cudaError_t e = tc_set_attributes();
    if (e != cudaSuccess) return e;
    tc_grad_kernel<<<grid, kGThreads, kGSmemBytes, s>>>(p);
    return cudaGetLastError();
}

cudaError_t tc_launch_knn(const TcArgs &a, dim3 grid, cudaStream_t s) {
    TcParams p;
    if (a.m_pad % kKRows || a.n_pad % kKCols || a.chunk % kKCols || a.D < 32 || a.D > 62 || a.K < 1 ||
        a.K > a.KP || !a.carry)
        return cudaErrorInvalidValue;
    // the screen reads the high halves only: A tiles of 128 rows, B tiles of 128 points
    if (!make_map(&p.tm_a_hi, a.a_hi, a.m_pad, kRows) || !make_map(&p.tm_b_hi, a.b_hi, a.n_pad, kKCols))
        return cudaErrorInvalidValue;
    p.bpad = nullptr;
    p.fpad = nullptr;
    p.out = a.out;  // the distances (or null)
    p.ws0 = a.ws0;
    p.ws1 = nullptr;
    p.guard = a.guard;
    p.wait_ns = a.wait_ns;
    p.starve = a.starve ? 1 : 0;
    p.M = a.M;
    p.N = a.N;
    p.chunk = a.chunk;
    p.S = a.S;
    p.x = a.x;
    p.g = nullptr;
    p.D = a.D;
    p.c = 1.f;
    p.gscale = 0.f;
    p.flags = nullptr;
    p.y = a.y;
    p.idx = a.idx;
    p.wsi = a.wsi;
    p.K = a.K;
    p.carry = a.carry;
    cudaError_t e = tc_set_attributes();
    if (e != cudaSuccess) return e;
    switch (a.KP) {
        case 1: tc_knn_kernel<1><<<grid, kThreadsTc, kSmemBytes, s>>>(p); break;
        case 4: tc_knn_kernel<4><<<grid, kThreadsTc, kSmemBytes, s>>>(p); break;
        case 10: tc_knn_kernel<10><<<grid, kThreadsTc, kSmemBytes, s>>>(p); break;
        case 16: tc_knn_kernel<16><<<grid, kThreadsTc, kSmemBytes, s>>>(p); break;
        case 32: tc_knn_kernel<32><<<grid, kThreadsTc, kSmemBytes, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

int tc_grad_occupancy() {
    int n = 0;
    if (tc_set_attributes() != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_grad_kernel, kGThreads, kGSmemBytes) != cudaSuccess)
        return 0;
    return n;
}

int tc_occupancy() {
    int n = 0;
    if (tc_set_attributes() != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_sum_kernel, kThreadsTc, kSmemBytes) != cudaSuccess)
        return 0;
    return n;
}

bool tc_available() { return encode_fn() != nullptr; }

cudaError_t tc_read_status(bool clear, unsigned *status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_tc_status, sizeof(unsigned));
    if (e == cudaSuccess && clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace kr
