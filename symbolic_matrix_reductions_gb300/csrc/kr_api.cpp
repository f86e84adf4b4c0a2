// kr_api.cpp -- the C ABI: argument validation, launch planning, host-buffer
// staging, stream-ordered workspace, launches.  No device code here.
//
// Planning: a launch is a grid of (row blocks, S) blocks.  A row block owns
// kThreads * R rows; S splits the j axis into S disjoint ranges whose partial
// results a second kernel combines in a fixed order (split-j).  S is chosen to
// minimise a model of the busiest SM's time: it runs ceil(blocks / SMs) blocks of
// (chunk + per-tile overhead [+ K-min insertions]) work each, at full rate when it
// holds at least 16 resident warps and proportionally slower below that, and (except
// K-min) a little slower the fewer waves of blocks there are.  So
// small-M / huge-N problems (the tall products of the GitHub issue "Transparent
// interface for billion-scale matrices") still fill every SM, the last wave of a
// large problem is not left mostly empty, and K-min, whose register list restarts
// in every split (early in a scan almost every point enters it), is split only
// when the extra parallelism pays for the extra insertions.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "kr_config.h"
#include "kr_internal.h"
#include "kr_tc.h"

namespace kr {

static thread_local int g_last_cuda_error = 0;

static int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return KR_ERR_CUDA;
}

Instance choose_instance(int op, int D, int EK, int kind) {
    Instance in{};
    in.d_pad = pad_d(D);
    if (op == OP_KNN) {
        in.ek_pad = pad_k(EK);
        in.rows = rows_knn(in.d_pad, in.ek_pad);
        in.tile = knn_instance_tile(in.d_pad);
    } else {
        in.ek_pad = pad_e(EK);
        in.rows = (op == OP_GRAD) ? (wide_grad(in.d_pad) ? 1 : rows_grad(in.d_pad, in.ek_pad))
                                  : rows_fwd(in.d_pad, in.ek_pad);
        in.tile = (op == OP_GRAD && wide_grad(in.d_pad))    ? kWideGradTile
                  : (op == OP_GRAD && !packed_grad(in.d_pad)) ? tile_points(pack_stride(in.d_pad, in.ek_pad))
                                                              : instance_tile(in.d_pad, in.ek_pad);
        in.rec = streamed(in.d_pad) && (op == OP_LSE || op == OP_GRAD || (op == OP_SUM && kind == KR_KERNEL_GAUSSIAN));
    }
    return in;
}

static int64_t round256(int64_t v) { return (v + 255) / 256 * 256; }

// Bytes of the streamed records (and LogSumExp tile frames) of a call with N points.
static int64_t record_bytes(int op, const Instance &in, int64_t N, int64_t batch) {
    if (!in.rec) return 0;
    return batch * (round256(record_elems(in, N) * (int64_t)sizeof(float)) +
                    round256(wtile_elems(op, in, N) * (int64_t)sizeof(float)));
}

// Bytes of split-j workspace for S splits.
static int64_t workspace_bytes(int op, const Instance &in, int64_t M, int D, int EK, int S) {
    if (S <= 1) return 0;
    switch (op) {
        case OP_SUM:
        case OP_LSE: return 2 * (int64_t)S * M * EK * (int64_t)sizeof(float);
        case OP_GRAD: return 2 * (int64_t)S * M * D * (int64_t)sizeof(float);
        case OP_KNN: return (int64_t)S * M * in.ek_pad * (int64_t)(sizeof(float) + sizeof(int32_t));
        case OP_MAX: return (int64_t)S * M * EK * (int64_t)(sizeof(float) + sizeof(int32_t));
    }
    return 0;
}

static const int64_t kMaxWorkspace = (int64_t)1 << 30;  // 1 GiB of partials at most

static const int64_t kMaxTcOperands = (int64_t)8 << 30;  // split fp16 operands of the tensor path
static const int64_t kTcChunkMax = (int64_t)3 << 16;     // points per tensor-path split: 48 MB of B operands

static int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Tensor-core plan: kTcRows rows per block (one TMEM lane each), tiles of kTcCols points
// (the x-gradient: kTcGradCols; the K-min: kTcKnnRows rows, tiles of kTcKnnCols), splits on
// tile boundaries, one block per SM.  Split partials: M values (Sum, LSE), M x D (the
// gradient) or M lists (the K-min) per split.
static void plan_tc(int op, int64_t M, int64_t N, int D, int EK, int num_sms, int blocks_per_sm, int forced_split,
                    kr_plan_t *p) {
    const int tile = op == OP_GRAD ? kTcGradCols : op == OP_KNN ? kTcKnnCols : kTcCols;
    const int rows = op == OP_KNN ? kTcKnnRows : kTcRows;  // rows a block
    // split partials per row: (hi, lo) of the Sum / LSE; D of them for the gradient; a list of
    // KP (distance, index) for the K-min (the same bytes: 2 x 4 a slot)
    const int64_t width = op == OP_GRAD ? D : op == OP_KNN ? pad_k(EK) : 1;
    p->d_pad = 64;
    p->ek_pad = op == OP_KNN ? pad_k(EK) : 1;
    p->rows_per_thread = 1;
    p->threads = op == OP_GRAD ? kTcGradThreads : kTcThreads;
    p->tile_points = tile;
    p->row_blocks = (M + rows - 1) / rows;
    p->path = KR_PATH_TENSOR_CORES;
    if (num_sms < 1) num_sms = 1;
    if (blocks_per_sm < 1) blocks_per_sm = 1;
    const int64_t tiles_total = std::max<int64_t>(1, (N + tile - 1) / tile);
    int S = 1;
    if (forced_split >= 1) {
        S = (int)std::min<int64_t>(std::min<int64_t>(forced_split, tiles_total), kMaxSplit);
    } else if (N > 0) {
        // The blocks resident at one time mostly share a split and stream its B tiles
        // at slightly different paces; while a split's operands (256 B per point) fit
        // in L2 every block after the first reads them from there.  Longer splits
        // fall out of L2 and the copy latency of the misses stalls the MMAs.
        // The partials cap the splits too (the gradient's are D times larger): when L2 residency
        // asks for more splits than the cap allows, take as many as it allows.
        const int64_t s_cap = std::max<int64_t>(
            1, std::min<int64_t>(std::min<int64_t>(kMaxSplit, tiles_total),
                                 kMaxWorkspace / std::max<int64_t>(1, 2 * M * width * (int64_t)sizeof(float))));
        const int64_t min_split = std::min<int64_t>((N + kTcChunkMax - 1) / kTcChunkMax, s_cap);
        // per block: its tiles plus a fixed start-up cost of about 1/8 tile
        double best = 0.0;
        for (int64_t s = std::max<int64_t>(1, min_split); s <= s_cap; ++s) {
            const int64_t chunk = round_up((N + s - 1) / s, tile);
            const double work = (double)(chunk / tile) + 0.125;
            const int64_t per_sm = (p->row_blocks * s + num_sms - 1) / num_sms;
            const double cost = (double)per_sm * work * (1.0 + 0.002 * (double)s);
            if (best == 0.0 || cost < best * 0.999) {
                best = cost;
                S = (int)s;
            }
        }
    }
    p->chunk = round_up((std::max<int64_t>(N, 1) + S - 1) / S, tile);
    S = (int)std::max<int64_t>(1, (N + p->chunk - 1) / p->chunk);  // every split nonempty
    p->split = S;
    const int64_t n_pad = round_up(std::max<int64_t>(N, 1), kTcCols);
    // split fp16 operands (256 B a point), the padded signal / weights, the LSE tile frames
    const int64_t operands = (round_up(std::max<int64_t>(M, 1), rows) + n_pad) * 256 + n_pad * 4 +
                             round_up(n_pad / kTcCols * 4, 256);
    p->workspace_bytes = 256 + operands + (S > 1 ? 2 * (int64_t)S * M * width * (int64_t)sizeof(float) : 0) +
                         (op == OP_GRAD ? round_up((int64_t)S * M, 256) : 0) +  // the gradient's weak-row flags
                         (op == OP_KNN ? round_up(4 * M * width, 256) : 0);      // the K-min's shared lists
}

static int64_t batch_of(const kr_options *opt) { return opt && opt->batch > 1 ? opt->batch : 1; }

static bool tc_eligible(int op, int64_t M, int64_t N, int D, int EK, const kr_options *opt) {
    const int path = opt ? opt->path : 0, kind = opt ? opt->kernel : KR_KERNEL_GAUSSIAN;
    if (path == KR_PATH_CUDA_CORES) return false;
    if (op == OP_KNN) {  // the screen: the Sum's coordinate range, lists of up to 32
        if (!(D >= 32 && D <= 62 && EK >= 1 && EK <= 32) || batch_of(opt) > 1) return false;
    } else if ((op != OP_SUM && op != OP_LSE && op != OP_GRAD) || kind != KR_KERNEL_GAUSSIAN || !tc_dims(D, EK)) {
        return false;
    }
    if (op == OP_LSE && D > kTcLseMaxD) return false;  // the weight takes one more operand slot
    if (batch_of(opt) > 1) return false;  // the tensor-core prepass and tiles serve one problem
    return (round_up(std::max<int64_t>(M, 1), kTcRows) + round_up(std::max<int64_t>(N, 1), kTcCols)) * 256 <=
           kMaxTcOperands;
}

// Pure planner (no CUDA call).  blocks_per_sm <= 0: assume 4 resident blocks.  Streamed
// instances split on tile boundaries (every split's range is whole prepass tiles) and add
// their records to the workspace.
static int plan(int op, int64_t M, int64_t N, int D, int EK, int num_sms, int blocks_per_sm,
                int forced_split, int64_t batch, int kind, kr_plan_t *p) {
    Instance in = choose_instance(op, D, EK, kind);
    // Splits on whole tiles whether or not the call streams, so that the same split gives
    // the same tiles (and the same bits) either way; batched problems are small, and there a
    // prepass launch would cost more than streaming saves.
    const int64_t align = in.rec ? in.tile : 1;
    if (batch > 1) in.rec = false;
    p->path = KR_PATH_CUDA_CORES;
    p->d_pad = in.d_pad;
    p->ek_pad = in.ek_pad;
    p->rows_per_thread = in.rows;
    p->threads = kThreads;
    p->tile_points = in.tile;
    const int64_t bm = (int64_t)kThreads * in.rows;
    p->row_blocks = (M + bm - 1) / bm;
    if (num_sms < 1) num_sms = 1;
    if (blocks_per_sm < 1) blocks_per_sm = 4;

    int S = 1;
    if (forced_split >= 1) {
        S = (int)std::min<int64_t>(forced_split, std::max<int64_t>(N, 1));
        S = std::min(S, kMaxSplit);
    } else if (N > 0 && p->row_blocks > 0) {
        // At least 64 points per split, at most kMaxSplit splits.
        const int64_t s_max = std::min<int64_t>(kMaxSplit, std::max<int64_t>(1, N / 64));
        // K-min: warp-level insertion events per row slot and split, each worth
        // `ins_points` points of distance work (about 75 instructions against
        // D + 1.25 per point and row for the packed kernel, 2D + 1 for the scalar).
        const bool pk = packed(in.d_pad);
        const double pt_cost = pk ? in.d_pad + 1.25 : 2.0 * in.d_pad + 1.0;
        const double ins_points = 75.0 / pt_cost;
        const double group = pk ? 2.0 * unroll_pairs(in.d_pad) : (double)unroll_points(in.d_pad);
        const double lanes_k = 32.0 * in.ek_pad;
        double best = 0.0;
        for (int64_t s = 1; s <= s_max; ++s) {
            if (batch * workspace_bytes(op, in, M, D, EK, (int)s) > kMaxWorkspace) break;
            const int64_t chunk = round_up((N + s - 1) / s, align);
            if (s > 1 && (s - 1) * chunk >= N) continue;  // an empty split: the same as fewer splits
            const int64_t tiles = (chunk + in.tile - 1) / in.tile;
            // per block, in points: its chunk, a per-tile cost (staging, barriers) and a fixed
            // cost (loading its rows, writing its partials, its share of the combine)
            double work = (double)chunk + 32.0 * (double)tiles + 128.0;
            if (op == OP_KNN) {
                const double groups = (double)chunk / group;
                const double events = groups <= lanes_k ? groups : lanes_k * (1.0 + std::log(groups / lanes_k));
                work += events * ins_points;
            }
            const int64_t per_sm = (p->row_blocks * s * batch + num_sms - 1) / num_sms;
            const int64_t conc = std::min<int64_t>(per_sm, blocks_per_sm);
            const double eff = std::min(1.0, (double)(conc * (kThreads / 32)) / 16.0);
            // Load balance: with few waves of large blocks the slowest SM sets the end; with
            // more, smaller blocks the faster SMs take more of them.  Fitted on forced-split
            // timings of the D = 3 x-gradient at M = N = 1e5 (3 splits, 0.97 waves, 7 % slower
            // than 10 splits, 3.2 waves).  K-min keeps its own insertion term instead (its
            // lists restart in every split).
            const double waves = (double)(p->row_blocks * s * batch) / ((double)num_sms * blocks_per_sm);
            const double balance = op == OP_KNN ? 1.0 : 1.0 + 0.136 / waves;
            // each split also costs a little in partial traffic and the combine, and splitting
            // at all costs a workspace allocation and a combine launch (worth ~4096 points of
            // one block's work, about 60 us)
            const double cost =
                (double)per_sm * work / eff * balance * (1.0 + 0.002 * (double)s) + (s > 1 ? 4096.0 : 0.0);
            if (s == 1 || cost < best * 0.999) {
                best = cost;
                S = (int)s;
            }
        }
    }
    p->split = S;
    p->chunk = round_up((N + S - 1) / S, align);
    if (p->chunk < 1) p->chunk = 1;
    // Every split must own a nonempty range, except when N == 0.
    if (N > 0 && (int64_t)(S - 1) * p->chunk >= N) {
        S = (int)((N + p->chunk - 1) / p->chunk);
        p->split = S;
    }
    const int64_t parts = batch * workspace_bytes(op, in, M, D, EK, S);
    p->workspace_bytes = in.rec ? round256(parts) + record_bytes(op, in, N, batch) : parts;
    return KR_OK;
}

// ---- per-device cached attributes -----------------------------------------------
namespace {
struct DeviceCache {
    int num_sms = 0;
    int occ[kNumOps][kNumKernels][10][33] = {};  // resident blocks per (op, kernel kind, d_pad index,
                                                 // ek_pad); 0 = not queried
    int tc_occ = 0;           // resident tensor-core Sum blocks; 0 = not queried
    cudaMemPool_t pool = nullptr;  // the library's workspace pool on this device
    bool pool_tried = false;
    unsigned *dbg = nullptr;       // debug builds: the index-check status word
};
std::mutex g_cache_mutex;
DeviceCache g_cache[64];

int d_index(int d_pad) {
    switch (d_pad) {
        case 1: case 2: case 3: case 4: return d_pad - 1;
        case 8: return 4;
        case 16: return 5;
        case 32: return 6;
        case 50: return 7;
        case 64: return 8;
        default: return 9;
    }
}

int occupancy_radial(int kind, int red, const Instance &in) {
    switch (kind) {
        case KR_KERNEL_GAUSSIAN: return occupancy_radial_gauss(red, in);
        case KR_KERNEL_LAPLACE: return occupancy_radial_laplace(red, in);
        case KR_KERNEL_CAUCHY: return occupancy_radial_cauchy(red, in);
        case KR_KERNEL_INVERSE_MULTIQUADRIC: return occupancy_radial_imq(red, in);
    }
    return 0;
}

int query_occupancy(int op, int kind, const Instance &in) {
    if (op == OP_MAX) return occupancy_radial(kind, 1, in);
    if (op == OP_SUM && kind != KR_KERNEL_GAUSSIAN) return occupancy_radial(kind, 0, in);
    switch (op) {
        case OP_SUM: return occupancy_sum(in);
        case OP_LSE: return occupancy_lse(in);
        case OP_GRAD: return occupancy_grad(in);
        case OP_KNN: return occupancy_knn(in);
    }
    return 0;
}

int device_info(int dev, int op, int kind, const Instance &in, int *num_sms, int *occ) {
    if (dev < 0 || dev >= 64) return -1;
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    DeviceCache &c = g_cache[dev];
    if (c.num_sms == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        c.num_sms = n;
    }
    *num_sms = c.num_sms;
    int &slot = c.occ[op][kind][d_index(in.d_pad)][in.ek_pad];
    if (slot == 0) slot = query_occupancy(op, kind, in);
    *occ = slot;
    return 0;
}

// Workspace and staging memory come from a stream-ordered pool the library owns on
// each device, so freed blocks are reused by the next call instead of going back to
// the driver at every synchronisation (the default pool's behaviour).  The pool keeps
// at most kPoolKeep bytes across synchronisations; larger peaks are returned.
constexpr uint64_t kPoolKeep = (uint64_t)256 << 20;

cudaMemPool_t device_pool(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    DeviceCache &c = g_cache[dev];
    if (!c.pool_tried) {
        c.pool_tried = true;
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
            uint64_t keep = kPoolKeep;
            cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
            c.pool = pool;
        } else {
            cudaGetLastError();  // no pool: allocate from the device's default pool
        }
    }
    return c.pool;
}

int device_tc_occupancy(int dev) {
    if (dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    if (g_cache[dev].tc_occ == 0) g_cache[dev].tc_occ = tc_occupancy();
    return g_cache[dev].tc_occ;
}
}  // namespace

// Debug builds (-DKR_DEBUG): the device word the kernels' index checks write to, one
// per device for the life of the process.  Release builds never allocate it.
unsigned *debug_word(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    DeviceCache &c = g_cache[dev];
    if (!c.dbg) {
        unsigned *p = nullptr;
        if (cudaMalloc((void **)&p, sizeof(unsigned)) == cudaSuccess && cudaMemset(p, 0, sizeof(unsigned)) == cudaSuccess)
            c.dbg = p;
        else
            cudaGetLastError();
    }
    return c.dbg;
}

// Bound of every mbarrier wait of the tensor-core kernels, in ms: KREDUCE_TC_WAIT_MS read
// once per process (2000 if unset or not positive), or what kr_set_tc_test_hooks set.
// Starvation of the B tiles (the failure-detection test) exists only in debug builds.
static std::once_flag g_tc_wait_once;
static std::atomic<long> g_tc_wait_ms{2000};
static std::atomic<int> g_tc_starve{0};

static uint64_t tc_wait_ns() {
    std::call_once(g_tc_wait_once, [] {
        const char *wms = std::getenv("KREDUCE_TC_WAIT_MS");
        const long ms = wms ? std::strtol(wms, nullptr, 10) : 0;
        if (ms > 0) g_tc_wait_ms.store(ms);
    });
    return (uint64_t)g_tc_wait_ms.load() * 1000000ull;
}

// ---- validation ---------------------------------------------------------------------
static bool overlaps(const void *a, int64_t abytes, const void *b, int64_t bbytes) {
    if (!a || !b || abytes <= 0 || bbytes <= 0) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

// Element counts up to 2^60, so that byte sizes (x 4 or 8) and every 64-bit element index
// stay far from overflow.
static bool fits_elements(int64_t rows, int64_t cols) {
    return rows >= 0 && cols >= 0 && (cols == 0 || rows <= ((int64_t)1 << 60) / cols);
}

struct Buf {
    const void *ptr;
    int64_t bytes;
    bool output;
};

static int validate(int op, const Buf *bufs, int nbuf, int64_t M, int64_t N, int D, int EK, float sigma,
                    const kr_options *opt) {
    if (M < 0 || N < 0) return KR_ERR_INVALID;
    if (D < 1 || EK < 1) return KR_ERR_INVALID;
    if (op != OP_KNN && !(std::isfinite(sigma) && sigma > 0.f)) return KR_ERR_INVALID;
    if (opt) {
        if (opt->split < 0) return KR_ERR_INVALID;
        if (opt->path < KR_PATH_AUTO || opt->path > KR_PATH_TENSOR_CORES) return KR_ERR_INVALID;
        if (opt->kernel < 0 || opt->kernel >= kNumKernels) return KR_ERR_INVALID;
        if (opt->batch < 0) return KR_ERR_INVALID;
        if (opt->batch > kMaxBatch) return KR_ERR_UNSUPPORTED;
        for (int k = 0; k < 4; ++k)
            if (opt->reserved[k] != 0) return KR_ERR_INVALID;
        // the other kernels serve the Sum (and the b-gradient) and Max / Min
        if (opt->kernel != KR_KERNEL_GAUSSIAN && op != OP_SUM && op != OP_MAX) return KR_ERR_UNSUPPORTED;
    }
    if (D > kMaxD) return KR_ERR_UNSUPPORTED;
    if (op == OP_KNN ? EK > kMaxK : EK > kMaxE) return KR_ERR_UNSUPPORTED;
    const int64_t Mx = std::max<int64_t>(M, 1), Nx = std::max<int64_t>(N, 1);
    if (!fits_elements(Mx, D) || !fits_elements(Nx, D) || !fits_elements(Mx, EK) || !fits_elements(Nx, EK))
        return KR_ERR_UNSUPPORTED;
    if (N > INT32_MAX - 1) return KR_ERR_UNSUPPORTED;
    for (int k = 0; k < nbuf; ++k)
        if (bufs[k].bytes > 0 && bufs[k].ptr == nullptr) return KR_ERR_INVALID;
    for (int k = 0; k < nbuf; ++k) {
        if (!bufs[k].output) continue;
        for (int l = 0; l < nbuf; ++l) {
            if (l == k) continue;
            if (overlaps(bufs[k].ptr, bufs[k].bytes, bufs[l].ptr, bufs[l].bytes)) return KR_ERR_INVALID;
        }
    }
    return KR_OK;
}

// ---- allocation (with an opt-in failure injection for tests) -----------------------
static cudaError_t ws_alloc(void **p, size_t bytes, cudaStream_t s, int dev) {
    // KREDUCE_FAIL_ALLOC=1 makes every workspace/staging allocation fail, so that
    // the KR_ERR_ALLOC path can be tested without exhausting device memory.
    const char *inj = std::getenv("KREDUCE_FAIL_ALLOC");
    if (inj && inj[0] == '1') {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    cudaMemPool_t pool = device_pool(dev);
    return pool ? cudaMallocFromPoolAsync(p, bytes, pool, s) : cudaMallocAsync(p, bytes, s);
}

// Is `p` directly usable by kernels?  Host memory (pageable or pinned) is staged.
static int is_device_ptr(const void *p, bool *dev) {
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return (int)e;
    }
    *dev = (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged);
    return 0;
}

// ---- radial-kernel family: one launcher per kernel kind ------------------------------
static cudaError_t launch_radial(int kind, int red, const Instance &in, const Args &a, dim3 grid,
                                 cudaStream_t s) {
    switch (kind) {
        case KR_KERNEL_GAUSSIAN: return launch_radial_gauss(red, in, a, grid, s);
        case KR_KERNEL_LAPLACE: return launch_radial_laplace(red, in, a, grid, s);
        case KR_KERNEL_CAUCHY: return launch_radial_cauchy(red, in, a, grid, s);
        case KR_KERNEL_INVERSE_MULTIQUADRIC: return launch_radial_imq(red, in, a, grid, s);
    }
    return cudaErrorInvalidValue;
}

// Coordinate prescale c of each kernel kind: the kernels evaluate k from |c x - c y|.
static double kernel_prescale(int kind, float sigma) {
    switch (kind) {
        case KR_KERNEL_LAPLACE: return 1.4426950408889634 / (double)sigma;     // 2^(-|x'-y'|)
        case KR_KERNEL_CAUCHY:
        case KR_KERNEL_INVERSE_MULTIQUADRIC: return 1.0 / (double)sigma;       // 1 + |x'-y'|^2
        default: return std::sqrt(1.4426950408889634) / (double)sigma;         // 2^(-|x'-y'|^2)
    }
}

// ---- tensor-core Sum: operand prepass, tensor kernel, CUDA-core stand-in, combine -------
// Workspace: [guard (2 x u32) + status | A_hi | A_lo | B_hi | B_lo | padded b | LSE frames |
// partials | the gradient's flags or the K-min's shared lists].  The CUDA-core kernel is
// always launched after the tensor kernel with the same splits; it returns at once unless
// the prepass found norms the expansion cannot serve.
static cudaError_t run_tc(int op, Args a, const kr_plan_t &p, const Instance &in, char *ws, cudaStream_t stream) {
    const bool lse = op == OP_LSE, grad = op == OP_GRAD, knn = op == OP_KNN;
    const int64_t width = grad ? a.D : knn ? p.ek_pad : 1;  // split partials per row
    const int64_t m_pad = round_up(a.M, knn ? kTcKnnRows : kTcRows), n_pad = round_up(std::max<int64_t>(a.N, 1), kTcCols);
    unsigned *guard = (unsigned *)ws;
    __half *a_hi = (__half *)(ws + 256);
    __half *a_lo = a_hi + m_pad * 64;
    __half *b_hi = a_lo + m_pad * 64;
    __half *b_lo = b_hi + n_pad * 64;
    float *bpad = (float *)(b_lo + n_pad * 64);
    float *fpad = bpad + n_pad;
    float *part = (float *)((char *)fpad + round_up(n_pad / kTcCols * 4, 256));
    // the x-gradient's flags (S x M bytes), or the K-min's shared lists (M x KP), follow the
    // split partials
    uint8_t *flags = (uint8_t *)(part + (p.split > 1 ? 2 * (int64_t)p.split * a.M * width : 0));
    float *carry = knn ? (float *)flags : nullptr;
    cudaError_t ce = cudaMemsetAsync(guard, 0, 256, stream);
    // (the K-min's screen reads the operands' high halves only)
    if (ce == cudaSuccess)
        ce = tc_launch_prep(a.x, a.M, m_pad, a.D, a.c, true, lse, a_hi, knn ? nullptr : a_lo, guard, nullptr, nullptr,
                            nullptr, stream, false, carry, knn ? (int)width : 0);
    if (ce == cudaSuccess && grad) ce = tc_launch_bmax(a.b, a.N, guard, stream);
    if (ce == cudaSuccess)
        ce = tc_launch_prep(a.y, a.N, n_pad, a.D, a.c, false, lse, b_hi, knn ? nullptr : b_lo, guard + 1,
                            knn ? nullptr : a.b, (lse || knn) ? nullptr : bpad, lse ? fpad : nullptr, stream, grad);
    if (p.split > 1) {
        a.ws0 = part;
        if (knn)  // the lists' distances, then their indices (as the CUDA-core K-min lays them out)
            a.wsi = (int32_t *)(part + (int64_t)p.split * a.M * width);
        else
            a.ws1 = part + (int64_t)p.split * a.M * width;
    }
    if (ce == cudaSuccess) {
        TcArgs t{};
        t.a_hi = a_hi;
        t.a_lo = a_lo;
        t.b_hi = b_hi;
        t.b_lo = b_lo;
        t.bpad = bpad;
        t.fpad = fpad;
        t.lse = lse;
        t.m_pad = m_pad;
        t.n_pad = n_pad;
        t.out = a.out;
        t.ws0 = a.ws0;
        t.ws1 = a.ws1;
        t.guard = guard;
        // Every mbarrier wait of the tensor kernel gives up after this long.  In debug builds
        // a test can withhold the B tiles (kr_set_tc_test_hooks) to watch the waits run out.
        t.wait_ns = tc_wait_ns();
#ifdef KR_DEBUG
        t.starve = g_tc_starve.load() != 0;
#else
        t.starve = false;
#endif
        t.M = a.M;
        t.N = a.N;
        t.chunk = p.chunk;
        t.S = p.split;
        t.x = a.x;
        t.g = a.g;
        t.D = a.D;
        t.c = a.c;
        t.gscale = a.gscale;
        t.flags = flags;
        t.y = a.y;
        t.idx = a.idx;
        t.wsi = a.wsi;
        t.K = a.K;
        t.KP = p.ek_pad;
        t.carry = carry;
        const dim3 tgrid((unsigned)p.row_blocks, (unsigned)p.split);
        ce = grad ? tc_launch_grad(t, tgrid, stream) : knn ? tc_launch_knn(t, tgrid, stream) : tc_launch_sum(t, tgrid, stream);
    }
    if (ce == cudaSuccess) {  // the CUDA-core stand-in: returns at once unless the guard failed
        a.tc_guard = guard;
        a.tc_flags = grad ? flags : nullptr;  // (or, for the gradient, on the rows flagged weak)
        const int64_t bm = (int64_t)kThreads * in.rows;
        const dim3 grid((unsigned)((a.M + bm - 1) / bm), (unsigned)p.split);
        ce = grad  ? launch_grad(in, a, grid, stream)
             : lse ? launch_lse(in, a, grid, stream)
             : knn ? launch_knn(in, a, grid, stream)
                   : launch_sum(in, a, grid, stream);
    }
    if (ce == cudaSuccess && p.split > 1) ce = launch_combine(op, in, a, stream);
    return ce;
}

// ---- the common driver --------------------------------------------------------------
// Block-sparse mode: the per-block work table and the column ranges, built on the host.
struct RangeTables {
    std::vector<int4> blocks;  // {first row, end row, first range, end range} per block
    std::vector<int2> ranges;  // column ranges [start, end)
    int64_t bytes() const { return (int64_t)(blocks.size() * sizeof(int4) + ranges.size() * sizeof(int2)); }
};

// Splits of the block-sparse mode: enough blocks for about two rounds of resident
// blocks on every SM, but every split keeps at least two tiles of the average block's
// ranges, and the partials stay within the workspace bound.
static int ranges_split(const RangeTables &rt, int tile, int num_sms, int occ, int64_t M, int EK) {
    if (rt.blocks.empty()) return 1;
    int64_t tiles = 0;
    for (const int4 &b : rt.blocks)
        for (int r = b.z; r < b.w; ++r) tiles += (rt.ranges[(size_t)r].y - rt.ranges[(size_t)r].x + tile - 1) / tile;
    const int64_t nb = (int64_t)rt.blocks.size();
    const int64_t target = 2 * (int64_t)std::max(num_sms, 1) * std::max(occ, 1);
    int64_t S = (target + nb - 1) / nb;
    S = std::min<int64_t>(S, std::max<int64_t>(1, tiles / (2 * nb)));
    S = std::min<int64_t>(S, kMaxSplit);
    while (S > 1 && 2 * S * M * EK * (int64_t)sizeof(float) > kMaxWorkspace) --S;
    return (int)std::max<int64_t>(S, 1);
}

static int run(int op, Buf *bufs, int nbuf, Args a, int EK, float sigma, cudaStream_t stream,
               const kr_options *opt, const RangeTables *rt = nullptr) {
    const int64_t B = batch_of(opt);
    // With a batch dimension every array holds B problems one after the other.
    for (int k = 0; k < nbuf; ++k) bufs[k].bytes *= B;
    int st = validate(op, bufs, nbuf, a.M, a.N, a.D, EK, sigma, opt);
    if (st != KR_OK) return st;
    if (a.M == 0) return KR_OK;

    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce);

    const int kind = opt ? opt->kernel : KR_KERNEL_GAUSSIAN;
    Instance in = choose_instance(op, a.D, EK, kind);
    int num_sms = 0, occ = 0;
    if (device_info(dev, op, kind, in, &num_sms, &occ) != 0) return cuda_fail(cudaGetLastError());
    kr_plan_t p;
    const bool tc = !rt && tc_eligible(op, a.M, a.N, a.D, EK, opt) && tc_available();
    // the tensor-core stand-in and the block-sparse kernels stage their own tiles, and so do
    // batched calls (small problems, where a prepass launch would cost more than it saves)
    if (tc || rt || B > 1) in.rec = false;
    if (tc) {
        plan_tc(op, a.M, a.N, a.D, EK, num_sms, device_tc_occupancy(dev), opt ? opt->split : 0, &p);
    } else {
        plan(op, a.M, a.N, a.D, EK, num_sms, occ, opt ? opt->split : 0, B, kind, &p);
        if (rt) {  // one block per table entry and split; the tables lead the workspace
            p.row_blocks = (int64_t)rt->blocks.size();
            p.split = ranges_split(*rt, in.tile, num_sms, occ, a.M, EK);
            p.chunk = std::max<int64_t>(a.N, 1);
            p.workspace_bytes = (rt->bytes() + 255) / 256 * 256 +
                                (p.split > 1 ? workspace_bytes(op, in, a.M, a.D, EK, p.split) : 0);
        }
    }
    {  // element counts of one problem's outputs and partials (index checks of debug builds)
        const int64_t w_out = op == OP_GRAD ? a.D : op == OP_KNN ? a.K : a.E;
        a.out_n = a.M * w_out;
        a.idx_n = a.M * (op == OP_KNN ? a.K : a.E);
        a.ws_n = (int64_t)p.split * a.M * (op == OP_GRAD ? a.D : op == OP_KNN ? p.ek_pad : a.E);
#ifdef KR_DEBUG
        a.dbg = debug_word(dev);
#endif
    }
    if (B > 1) {
        const int64_t w_out = op == OP_GRAD ? a.D : op == OP_KNN ? a.K : a.E;
        a.batch = (int)B;
        a.bs_x = a.M * a.D;
        a.bs_y = a.N * a.D;
        a.bs_b = a.N * a.E;
        a.bs_g = a.M * a.E;
        a.bs_out = a.M * w_out;
        a.bs_idx = a.M * (op == OP_KNN ? a.K : a.E);
        a.bs_ws = (int64_t)p.split * a.M * (op == OP_GRAD ? a.D : op == OP_KNN ? p.ek_pad : a.E);
    }

    // Host arrays: stage through one device allocation.
    bool host[8] = {};
    int64_t stage_bytes = 0;
    for (int k = 0; k < nbuf; ++k) {
        if (!bufs[k].ptr || bufs[k].bytes <= 0) continue;
        bool d = true;
        const int e = is_device_ptr(bufs[k].ptr, &d);
        if (e) return cuda_fail((cudaError_t)e);
        host[k] = !d;
        if (host[k]) stage_bytes += (bufs[k].bytes + 255) / 256 * 256;
    }
    const int64_t ws_bytes = (p.workspace_bytes + 255) / 256 * 256;
    char *mem = nullptr;
    if (stage_bytes + ws_bytes > 0) {
        ce = ws_alloc((void **)&mem, (size_t)(stage_bytes + ws_bytes), stream, dev);
        if (ce != cudaSuccess) {
            cudaGetLastError();
            return KR_ERR_ALLOC;
        }
    }
    void *dptr[8] = {};
    int64_t off = 0;
    int status = KR_OK;
    for (int k = 0; k < nbuf && status == KR_OK; ++k) {
        dptr[k] = const_cast<void *>(bufs[k].ptr);
        if (!host[k]) continue;
        dptr[k] = mem + off;
        off += (bufs[k].bytes + 255) / 256 * 256;
        if (!bufs[k].output) {
            ce = cudaMemcpyAsync(dptr[k], bufs[k].ptr, (size_t)bufs[k].bytes, cudaMemcpyHostToDevice, stream);
            if (ce != cudaSuccess) status = cuda_fail(ce);
        }
    }
    char *ws = mem ? mem + stage_bytes : nullptr;

    if (status == KR_OK) {
        // Buffer order: x, y, b, [g,] out | x, y, idx, dist | x, y, b, out, idx (Max)
        a.x = (const float *)dptr[0];
        a.y = (const float *)dptr[1];
        if (op == OP_KNN) {
            a.idx = (int32_t *)dptr[2];
            a.out = (float *)dptr[3];
        } else if (op == OP_MAX) {
            a.b = (const float *)dptr[2];
            a.out = (float *)dptr[3];
            a.idx = (int32_t *)dptr[4];
        } else {
            a.b = (const float *)dptr[2];
            if (op == OP_GRAD) {
                a.g = (const float *)dptr[3];
                a.out = (float *)dptr[4];
            } else {
                a.out = (float *)dptr[3];
            }
        }
        a.S = p.split;
        a.chunk = p.chunk;
        if (rt) {
            const size_t nb = rt->blocks.size() * sizeof(int4);
            ce = cudaMemcpyAsync(ws, rt->blocks.data(), nb, cudaMemcpyHostToDevice, stream);
            if (ce == cudaSuccess && !rt->ranges.empty())
                ce = cudaMemcpyAsync(ws + nb, rt->ranges.data(), rt->ranges.size() * sizeof(int2),
                                     cudaMemcpyHostToDevice, stream);
            a.blk = (const int4 *)ws;
            a.rng = (const int2 *)(ws + nb);
            if (p.split > 1) {  // split partials after the tables, laid out as in dense split-j
                char *part = ws + (rt->bytes() + 255) / 256 * 256;
                a.ws0 = (float *)part;
                if (op == OP_MAX)
                    a.wsi = (int32_t *)(part + (int64_t)p.split * a.M * EK * (int64_t)sizeof(float));
                else
                    a.ws1 = a.ws0 + (int64_t)p.split * a.M * EK;
            }
            if (ce == cudaSuccess)
                ce = launch_radial(kind, op == OP_MAX ? 1 : 0, in, a,
                                   dim3((unsigned)p.row_blocks, (unsigned)p.split, 1), stream);
            if (ce == cudaSuccess && p.split > 1) ce = launch_combine(op, in, a, stream);
        } else if (tc) {
            ce = run_tc(op, a, p, in, ws, stream);
        } else {
            const int64_t part_bytes = B * workspace_bytes(op, in, a.M, a.D, EK, p.split);
            if (p.split > 1) {
                a.ws0 = (float *)ws;
                if (op == OP_KNN) {
                    a.wsi = (int32_t *)(ws + B * p.split * a.M * p.ek_pad * (int64_t)sizeof(float));
                } else if (op == OP_MAX) {
                    a.wsi = (int32_t *)(ws + B * p.split * a.M * EK * (int64_t)sizeof(float));
                } else {
                    a.ws1 = (float *)(ws + part_bytes / 2);
                }
            }
            const dim3 grid((unsigned)p.row_blocks, (unsigned)p.split, (unsigned)B);
            if (in.rec && a.N > 0) {
                // the streamed instances: the prepass packs this call's tiles after the partials
                a.rec_n = record_elems(in, a.N);
                a.wtile_n = wtile_elems(op, in, a.N);
                a.bs_rec = round256(a.rec_n * (int64_t)sizeof(float)) / (int64_t)sizeof(float);
                a.bs_wtile = round256(a.wtile_n * (int64_t)sizeof(float)) / (int64_t)sizeof(float);
                a.rec = (float *)(ws + round256(part_bytes));
                a.wtile = op == OP_LSE ? a.rec + B * a.bs_rec : nullptr;
                ce = launch_pack(op, in, a, (a.N + in.tile - 1) / in.tile, stream);
            } else {
                in.rec = false;  // nothing to stream (N = 0): the kernel's own staging writes the empty result
            }
            if (ce == cudaSuccess) switch (op) {
                case OP_SUM:
                    ce = kind == KR_KERNEL_GAUSSIAN ? launch_sum(in, a, grid, stream)
                                                    : launch_radial(kind, 0, in, a, grid, stream);
                    break;
                case OP_MAX: ce = launch_radial(kind, 1, in, a, grid, stream); break;
                case OP_LSE: ce = launch_lse(in, a, grid, stream); break;
                case OP_GRAD: ce = launch_grad(in, a, grid, stream); break;
                default: ce = launch_knn(in, a, grid, stream); break;
            }
            if (ce == cudaSuccess && p.split > 1) ce = launch_combine(op, in, a, stream);
        }
        if (ce != cudaSuccess) status = cuda_fail(ce);
    }
    if (status == KR_OK) {
        for (int k = 0; k < nbuf; ++k) {
            if (!host[k] || !bufs[k].output) continue;
            ce = cudaMemcpyAsync(const_cast<void *>(bufs[k].ptr), dptr[k], (size_t)bufs[k].bytes,
                                 cudaMemcpyDeviceToHost, stream);
            if (ce != cudaSuccess) {
                status = cuda_fail(ce);
                break;
            }
        }
    }
    if (mem) {
        ce = cudaFreeAsync(mem, stream);
        if (ce != cudaSuccess && status == KR_OK) status = cuda_fail(ce);
    }
    if (stage_bytes > 0) {
        ce = cudaStreamSynchronize(stream);
        if (ce != cudaSuccess && status == KR_OK) status = cuda_fail(ce);
    }
    return status;
}

}  // namespace kr

using namespace kr;

extern "C" {

// Max / Min with their Arg: out (nullable when idx is given) and idx (nullable).
static int reduce_maxmin(const float *x, const float *y, const float *b, float *out, int32_t *idx, int64_t M,
                         int64_t N, int D, int E, float sigma, int reduction, kr_stream_t stream,
                         const kr_options *opt) {
    if (M < 0 || N < 0 || D < 1 || E < 1) return KR_ERR_INVALID;
    if (!out && !idx && M > 0) return KR_ERR_INVALID;
    const int64_t f = (int64_t)sizeof(float);
    Buf bufs[5] = {{x, M * D * f, false}, {y, N * D * f, false}, {b, N * E * f, false},
                   {out, out ? M * E * f : 0, true}, {idx, idx ? M * E * (int64_t)sizeof(int32_t) : 0, true}};
    Args a{};
    a.M = M;
    a.N = N;
    a.D = D;
    a.E = E;
    a.c = (float)kernel_prescale(opt ? opt->kernel : 0, sigma);
    a.vsign = reduction == KR_MAX ? 1.f : -1.f;
    return run(OP_MAX, bufs, 5, a, E, sigma, (cudaStream_t)stream, opt);
}

int kernel_reduce_ex(const float *x, const float *y, const float *b, float *out, int64_t M, int64_t N,
                     int D, int E, float sigma, int reduction, kr_stream_t stream, const kr_options *opt) {
    if (reduction == KR_MAX || reduction == KR_MIN) {
        if (!out && M > 0) return KR_ERR_INVALID;
        return reduce_maxmin(x, y, b, out, nullptr, M, N, D, E, sigma, reduction, stream, opt);
    }
    if (reduction != KR_SUM && reduction != KR_LSE) return KR_ERR_INVALID;
    const int op = reduction == KR_SUM ? OP_SUM : OP_LSE;
    if (M < 0 || N < 0 || D < 1 || E < 1) return KR_ERR_INVALID;
    const int64_t f = (int64_t)sizeof(float);
    Buf bufs[4] = {{x, M * D * f, false}, {y, N * D * f, false}, {b, N * E * f, false}, {out, M * E * f, true}};
    Args a{};
    a.M = M;
    a.N = N;
    a.D = D;
    a.E = E;
    a.K = 0;
    a.c = (float)kernel_prescale(op == OP_SUM && opt ? opt->kernel : 0, sigma);
    return run(op, bufs, 4, a, E, sigma, (cudaStream_t)stream, opt);
}

int kernel_reduce_arg_ex(const float *x, const float *y, const float *b, float *out, int32_t *idx, int64_t M,
                         int64_t N, int D, int E, float sigma, int reduction, kr_stream_t stream,
                         const kr_options *opt) {
    if (reduction != KR_MAX && reduction != KR_MIN) return KR_ERR_INVALID;
    if (!idx && M > 0) return KR_ERR_INVALID;
    return reduce_maxmin(x, y, b, out, idx, M, N, D, E, sigma, reduction, stream, opt);
}

int kernel_reduce_arg(const float *x, const float *y, const float *b, float *out, int32_t *idx, int64_t M,
                      int64_t N, int D, int E, float sigma, int reduction, kr_stream_t stream) {
    return kernel_reduce_arg_ex(x, y, b, out, idx, M, N, D, E, sigma, reduction, stream, nullptr);
}

int kernel_reduce_ranges(const float *x, const float *y, const float *b, float *out, int32_t *idx, int64_t M,
                         int64_t N, int D, int E, float sigma, int reduction, int64_t nclusters,
                         const int64_t *ranges_i, const int64_t *slices_i, int64_t nranges,
                         const int64_t *redranges_j, kr_stream_t stream, const kr_options *opt) {
    if (reduction != KR_SUM && reduction != KR_MAX && reduction != KR_MIN) return KR_ERR_INVALID;
    if (M < 0 || N < 0 || D < 1 || E < 1 || nclusters < 0 || nranges < 0) return KR_ERR_INVALID;
    if ((nclusters > 0 && (!ranges_i || !slices_i)) || (nranges > 0 && !redranges_j)) return KR_ERR_INVALID;
    if (reduction == KR_SUM ? (!out || idx) : (!out && !idx)) {
        if (M > 0) return KR_ERR_INVALID;
    }
    if (opt && (opt->split > 1 || opt->batch > 1)) return KR_ERR_UNSUPPORTED;
    // the tables: clusters disjoint and inside [0, M), slices non-decreasing, ranges inside [0, N)
    std::vector<int64_t> order((size_t)nclusters);
    for (int64_t c = 0; c < nclusters; ++c) {
        const int64_t i0 = ranges_i[2 * c], i1 = ranges_i[2 * c + 1];
        if (i0 < 0 || i1 < i0 || i1 > M) return KR_ERR_INVALID;
        if (slices_i[c] < (c ? slices_i[c - 1] : 0) || slices_i[c] > nranges) return KR_ERR_INVALID;
        order[(size_t)c] = c;
    }
    std::sort(order.begin(), order.end(), [&](int64_t p, int64_t q) { return ranges_i[2 * p] < ranges_i[2 * q]; });
    for (size_t k = 1; k < order.size(); ++k)
        if (ranges_i[2 * order[k]] < ranges_i[2 * order[k - 1] + 1]) return KR_ERR_INVALID;  // overlapping clusters
    RangeTables rt;
    rt.ranges.resize((size_t)nranges);
    for (int64_t r = 0; r < nranges; ++r) {
        const int64_t j0 = redranges_j[2 * r], j1 = redranges_j[2 * r + 1];
        if (j0 < 0 || j1 < j0 || j1 > N) return KR_ERR_INVALID;
        rt.ranges[(size_t)r] = make_int2((int)j0, (int)j1);
    }
    const int op = reduction == KR_SUM ? OP_SUM : OP_MAX;
    const int64_t bm = (int64_t)kThreads * choose_instance(op, D, E).rows;
    auto add_rows = [&](int64_t i0, int64_t i1, int r0, int r1) {
        for (int64_t i = i0; i < i1; i += bm)
            rt.blocks.push_back(make_int4((int)i, (int)std::min(i1, i + bm), r0, r1));
    };
    int64_t cursor = 0;
    for (int64_t c : order) {
        add_rows(cursor, ranges_i[2 * c], 0, 0);  // rows in no cluster: the empty reduction
        add_rows(ranges_i[2 * c], ranges_i[2 * c + 1], (int)(c ? slices_i[c - 1] : 0), (int)slices_i[c]);
        cursor = ranges_i[2 * c + 1];
    }
    add_rows(cursor, M, 0, 0);

    const int64_t f = (int64_t)sizeof(float);
    Buf bufs[5] = {{x, M * D * f, false}, {y, N * D * f, false}, {b, N * E * f, false},
                   {out, out ? M * E * f : 0, true}, {idx, idx ? M * E * (int64_t)sizeof(int32_t) : 0, true}};
    Args a{};
    a.M = M;
    a.N = N;
    a.D = D;
    a.E = E;
    a.c = (float)kernel_prescale(opt ? opt->kernel : 0, sigma);
    a.vsign = reduction == KR_MIN ? -1.f : 1.f;
    return run(op, bufs, 5, a, E, sigma, (cudaStream_t)stream, opt, &rt);
}

int kernel_reduce(const float *x, const float *y, const float *b, float *out, int64_t M, int64_t N, int D,
                  int E, float sigma, int reduction, kr_stream_t stream) {
    return kernel_reduce_ex(x, y, b, out, M, N, D, E, sigma, reduction, stream, nullptr);
}

int kernel_reduce_grad_x_ex(const float *x, const float *y, const float *b, const float *g, float *gx,
                            int64_t M, int64_t N, int D, int E, float sigma, kr_stream_t stream,
                            const kr_options *opt) {
    if (M < 0 || N < 0 || D < 1 || E < 1) return KR_ERR_INVALID;
    const int64_t f = (int64_t)sizeof(float);
    Buf bufs[5] = {{x, M * D * f, false}, {y, N * D * f, false}, {b, N * E * f, false},
                   {g, M * E * f, false}, {gx, M * D * f, true}};
    Args a{};
    a.M = M;
    a.N = N;
    a.D = D;
    a.E = E;
    const double c = std::sqrt(1.4426950408889634) / (double)sigma;
    a.c = (float)c;
    a.gscale = (float)(-2.0 / ((double)sigma * (double)sigma * c));
    return run(OP_GRAD, bufs, 5, a, E, sigma, (cudaStream_t)stream, opt);
}

int kernel_reduce_grad_x(const float *x, const float *y, const float *b, const float *g, float *gx, int64_t M,
                         int64_t N, int D, int E, float sigma, kr_stream_t stream) {
    return kernel_reduce_grad_x_ex(x, y, b, g, gx, M, N, D, E, sigma, stream, nullptr);
}

// The y-gradient is the x-gradient kernel with the clouds' roles exchanged: with
// X = y, Y = x, B = g, G = b it computes -(2/sigma^2) sum_i k_ij (sum_e b_je g_ie)
// (y_jd - x_id), which is d/dy_jd of sum_ie g_ie a_ie.
int kernel_reduce_grad_y_ex(const float *x, const float *y, const float *b, const float *g, float *gy,
                            int64_t M, int64_t N, int D, int E, float sigma, kr_stream_t stream,
                            const kr_options *opt) {
    if (M < 0 || N < 0 || D < 1 || E < 1) return KR_ERR_INVALID;
    const int64_t f = (int64_t)sizeof(float);
    Buf bufs[5] = {{y, N * D * f, false}, {x, M * D * f, false}, {g, M * E * f, false},
                   {b, N * E * f, false}, {gy, N * D * f, true}};
    Args a{};
    a.M = N;
    a.N = M;
    a.D = D;
    a.E = E;
    const double c = std::sqrt(1.4426950408889634) / (double)sigma;
    a.c = (float)c;
    a.gscale = (float)(-2.0 / ((double)sigma * (double)sigma * c));
    return run(OP_GRAD, bufs, 5, a, E, sigma, (cudaStream_t)stream, opt);
}

int kernel_reduce_grad_y(const float *x, const float *y, const float *b, const float *g, float *gy, int64_t M,
                         int64_t N, int D, int E, float sigma, kr_stream_t stream) {
    return kernel_reduce_grad_y_ex(x, y, b, g, gy, M, N, D, E, sigma, stream, nullptr);
}

// The b-gradient sum_i k_ij g_ie is the Sum reduction over i of the exchanged clouds
// (the Gaussian is symmetric in its two points).
int kernel_reduce_grad_b_ex(const float *x, const float *y, const float *g, float *gb, int64_t M, int64_t N,
                            int D, int E, float sigma, kr_stream_t stream, const kr_options *opt) {
    return kernel_reduce_ex(y, x, g, gb, N, M, D, E, sigma, KR_SUM, stream, opt);
}

int kernel_reduce_grad_b(const float *x, const float *y, const float *g, float *gb, int64_t M, int64_t N, int D,
                         int E, float sigma, kr_stream_t stream) {
    return kernel_reduce_grad_b_ex(x, y, g, gb, M, N, D, E, sigma, stream, nullptr);
}

int kernel_knn_ex(const float *x, const float *y, int32_t *idx, float *dist, int64_t M, int64_t N, int D,
                  int K, kr_stream_t stream, const kr_options *opt) {
    if (M < 0 || N < 0 || D < 1 || K < 1) return KR_ERR_INVALID;
    const int64_t f = (int64_t)sizeof(float);
    Buf bufs[4] = {{x, M * D * f, false}, {y, N * D * f, false}, {idx, M * K * (int64_t)sizeof(int32_t), true},
                   {dist, dist ? M * K * f : 0, true}};
    Args a{};
    a.M = M;
    a.N = N;
    a.D = D;
    a.E = 1;
    a.K = K;
    a.c = 1.f;
    return run(OP_KNN, bufs, 4, a, K, 1.f, (cudaStream_t)stream, opt);
}

int kernel_knn(const float *x, const float *y, int32_t *idx, float *dist, int64_t M, int64_t N, int D, int K,
               kr_stream_t stream) {
    return kernel_knn_ex(x, y, idx, dist, M, N, D, K, stream, nullptr);
}

const char *kr_status_string(int status) {
    switch (status) {
        case KR_OK: return "ok";
        case KR_ERR_INVALID: return "invalid argument";
        case KR_ERR_UNSUPPORTED: return "unsupported size or shape";
        case KR_ERR_ALLOC: return "workspace allocation failed";
        case KR_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

int kr_last_cuda_error(void) { return g_last_cuda_error; }

int kr_device_status(unsigned *status, int clear) {
    if (!status) return KR_ERR_INVALID;
    *status = 0;
    if (!tc_available()) return KR_OK;  // no device work can have run
    cudaError_t e = tc_read_status(clear != 0, status);
#ifdef KR_DEBUG
    int dev = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    unsigned *w = e == cudaSuccess ? debug_word(dev) : nullptr;
    if (w) {
        unsigned v = 0;
        e = cudaMemcpy(&v, w, sizeof(unsigned), cudaMemcpyDeviceToHost);
        if (e == cudaSuccess && clear) e = cudaMemset(w, 0, sizeof(unsigned));
        *status |= v << 8;
    }
#endif
    return e == cudaSuccess ? KR_OK : cuda_fail(e);
}

int kr_set_tc_test_hooks(int wait_ms, int starve) {
    if (wait_ms < 0 || (starve != 0 && starve != 1)) return KR_ERR_INVALID;
#ifndef KR_DEBUG
    if (starve) return KR_ERR_UNSUPPORTED;  // release builds carry no fault path
#endif
    tc_wait_ns();  // the environment's default is read first, so it cannot override this call
    g_tc_wait_ms.store(wait_ms > 0 ? (long)wait_ms : 2000);
    g_tc_starve.store(starve);
    return KR_OK;
}

int kr_debug_build(void) {
#ifdef KR_DEBUG
    return 1;
#else
    return 0;
#endif
}

int kr_plan(int op, int64_t M, int64_t N, int D, int EK, int num_sms, int blocks_per_sm, const kr_options *opt,
            kr_plan_t *out) {
    if (!out || op < 0 || op >= kNumOps) return KR_ERR_INVALID;
    const int st = validate(op, nullptr, 0, M, N, D, EK, 1.f, opt);
    if (st != KR_OK) return st;
    if (tc_eligible(op, M, N, D, EK, opt)) {
        plan_tc(op, M, N, D, EK, num_sms, blocks_per_sm, opt ? opt->split : 0, out);
        return KR_OK;
    }
    return plan(op, M, N, D, EK, num_sms, blocks_per_sm, opt ? opt->split : 0, batch_of(opt),
                opt ? opt->kernel : KR_KERNEL_GAUSSIAN, out);
}

int kr_plan_device(int op, int64_t M, int64_t N, int D, int EK, const kr_options *opt, kr_plan_t *out) {
    if (!out || op < 0 || op >= kNumOps) return KR_ERR_INVALID;
    const int st = validate(op, nullptr, 0, M, N, D, EK, 1.f, opt);
    if (st != KR_OK) return st;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce);
    int num_sms = 0, occ = 0;
    const int kind = opt ? opt->kernel : KR_KERNEL_GAUSSIAN;
    if (device_info(dev, op, kind, choose_instance(op, D, EK, kind), &num_sms, &occ) != 0)
        return cuda_fail(cudaGetLastError());
    if (tc_eligible(op, M, N, D, EK, opt) && tc_available()) {
        plan_tc(op, M, N, D, EK, num_sms, device_tc_occupancy(dev), opt ? opt->split : 0, out);
        return KR_OK;
    }
    return plan(op, M, N, D, EK, num_sms, occ, opt ? opt->split : 0, batch_of(opt), kind, out);
}

}  // extern "C"
