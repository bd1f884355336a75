// Exact scaled-dot-product attention forward for B300 (sm_103a).
//
// What is computed (see include/attn_api.h for the full statement and the pages it
// follows): O = softmax(scale * Q K^T + mask) V per (batch, query head), with the
// grouped-query head map kv = hq / (Hq / Hkv), the look-ahead mask j <= i and the
// causal sliding window i - j < W, plus the natural-log log-sum-exp of every row.
//
// How (one persistent kernel, one CTA per SM, 12 warps):
//   warps 0-3   softmax warpgroup for query tile 0 of the work unit (one row per thread)
//   warps 4-7   softmax warpgroup for query tile 1
//   warp 8      TMA producer: Q tiles once per unit, then K_j, V_j through a ring of
//               shared-memory stages guarded by full/empty mbarriers
//   warp 9      tensor-memory owner and MMA issuer: S_t = Q_t K_j^T into tensor memory,
//               then O_t += P_t V_j with P_t read from tensor memory
//   (warps 8 and 9 run their loops on all lanes with warp-uniform values and issue
//   each copy, MMA and commit from one lane elected inside the instruction's asm)
//   warps 10-11 idle; with warps 8-9 they form the warpgroup that hands registers to
//               the softmax warpgroups (setmaxnreg)
// A work unit is two consecutive 128-row query tiles of one (batch, query head); both
// tiles share every K/V tile the unit streams, so each K/V tile staged in shared
// memory feeds two MMAs. The two softmax warpgroups alternate with the tensor core:
// while one turns S into P, the tensor core runs the other tile's S and PV products.
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   [0,128) S0 / P0   [128,256) S1 / P1   [256,256+D) O0   [256+D,256+2D) O1
// P (bf16, two per column) overwrites the first half of its S block.
//
// Online softmax (the statistics of FlashAttention-2 kept on chip, as the
// FlashAttention-3 review page describes for FA1/FA2): per row a running maximum m
// (in log2 units of scale*s) and a running sum l. m is only raised when a tile's row
// maximum exceeds it by more than 8 (a factor 256), so P <= 256 and O is rescaled
// rarely; the result is exact because the final normalisation uses the same m.
//
// Every mbarrier wait is bounded in time; a wait that runs out sets a device status
// word, and the kernel drains its own copies and MMAs, frees its tensor memory and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_api.h"
#include "ptx.cuh"

namespace attn {

constexpr int BM = 128;  // query rows per tile = tensor-memory lanes
constexpr int BN = 128;  // keys per K/V tile
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 384;  // 3 warpgroups; warps 10-11 only hold registers back
// Register split: the kernel launches at LAUNCH_REGS per thread; the producer/MMA
// warpgroup gives registers back and the two softmax warpgroups take them, so that
// 2 * 128 * SOFTMAX_REGS + 128 * PRODUCER_REGS equals the launch total exactly.
constexpr int LAUNCH_REGS = 168;
constexpr int PRODUCER_REGS = 72;
constexpr int SOFTMAX_REGS = 216;
static_assert(2 * 128 * SOFTMAX_REGS + 128 * PRODUCER_REGS <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t STATUS_TIMEOUT = 1u;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
constexpr float LN2 = 0.693147180559945309f;
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s per wait
constexpr uint32_t WAIT_SLEEP_NS = 200000u;  // a waiting thread re-checks at least this often

__device__ unsigned int g_status;  // bit 0: some wait ran out of time; bit 1: an index check failed
constexpr uint32_t STATUS_BOUNDS = 2u;

// Index checks of the debug build (compiled with -DATTN_DEBUG). Each guards an access
// whose index comes from the scheduling arithmetic: a shared-memory stage or buffer,
// a tensor-memory column range, a tensor-map coordinate, a global row. A failed check
// sets bit 1 of the status word and records the first failing site; the caller then
// skips the access (a skipped copy leaves its barrier incomplete, and the bounded wait
// behind it ends the kernel). In the release build every check is the constant true
// and costs nothing.
#ifdef ATTN_DEBUG
__device__ unsigned int g_debug_site;
__device__ __noinline__ void debug_fail(unsigned int site) {
    atomicOr(&g_status, STATUS_BOUNDS);
    atomicCAS(&g_debug_site, 0u, site);
}
#define ATTN_CHECK(cond, site) ((cond) ? true : (::attn::debug_fail(site), false))
#else
#define ATTN_CHECK(cond, site) true
#endif

// Scratch of attn_fwd_decode_noalloc: the per-split partial results that attn_fwd_decode
// keeps in a caller-provided workspace live here instead, in a fixed array that every
// device holds from the moment it loads this library until the process exits. Host code
// must not use the name as a device address: the address comes from
// cudaGetSymbolAddress, taken once per device.
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(8) << 20;  // 8 MiB
static_assert(NOALLOC_SCRATCH_BYTES == ATTN_DECODE_NOALLOC_SCRATCH_BYTES,
              "the scratch size must match the limit the header states");
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Division of a non-negative int below 2^31 by an invariant divisor d >= 1, by a
// multiply-high and a shift (Granlund and Montgomery, "Division by invariant integers
// using multiplication", 1994, unsigned case): with l = ceil(log2 d) and
// mul = floor(2^32 (2^l - d) / d) + 1, the quotient is (mulhi(mul, n) + n) >> l.
// The sum stays below 2^32 because mulhi(mul, n) <= n < 2^31.
struct FastDiv {
    uint32_t mul, shift;
};

__host__ inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    FastDiv f;
    f.mul = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1ull);
    f.shift = l;
    return f;
}

__device__ __forceinline__ int fdiv(int n, FastDiv f) {
    const uint32_t un = static_cast<uint32_t>(n);
    return static_cast<int>((__umulhi(un, f.mul) + un) >> f.shift);
}

struct Params {
    __nv_bfloat16 *o;
    float *lse;
    const int *key_len;  // valid (unpadded) length per batch, or null: all N valid
    int B, Hq, Hkv, N, group;
    int causal, window;  // window 0 = none (a window >= N is passed as 0)
    int sym;             // window without the look-ahead mask: |i - j| < window
    int n_pairs, n_kv, num_units;
    float sl2;  // scale * log2(e)
    unsigned long long timeout_ns;
    FastDiv div_bh, div_hq, div_group;  // by B * Hq, Hq and Hq / Hkv
    // key-side length and query offset: keys per head Nk (= N except in the decode
    // shape), and query row i stands at position i + pos_off
    int Nk, pos_off;
    // decode shape: query tiles pack the G * Nq rows of one KV head (N = G * Nq rows
    // per tensor-map z index); unit = (batch * Hkv + hkv, split of the key tiles)
    int Nq, splits, split_lo, split_len, split_hi;
    // decode shape with both query tiles on one split (at most 32 packed rows): tile 0
    // takes the split's even key tiles, tile 1 the odd ones, over the same packed rows;
    // tile 1 hands its result to tile 0 through shared memory, which merges the two
    int dec2;
    FastDiv div_splits, div_nq;
    float *o_part, *lse_part;  // partial results per split (splits > 1), fp32
    float *o32;                // plain forward: O as fp32 instead of bf16 (null: bf16 to o)
    // e4m3 operands: per-block scales [z index][ceil(N / 128)] of Q, K and V
    const float *q_scale, *k_scale, *v_scale;
};

// F8: Q, K and V are e4m3 codes (1 byte) instead of bf16 (2 bytes); O stays bf16.
// DEC: the decode shape, which loads no Q for tile 1: its Q buffers have one slot, and at
// d = 128 the ring has room for two more stages.
template <int D, bool F8 = false, bool DEC = false>
struct Cfg {
    static constexpr int ELEM = F8 ? 1 : 2;                 // bytes per Q/K/V element
    static constexpr int KSTEP = F8 ? 32 : 16;              // reduction length of one MMA
    static constexpr int CHUNK_COLS = 128 / ELEM;           // columns of one 128-byte swizzled row
    static constexpr int CHUNK_BYTES = BM * 128;            // one slab: 128 rows x 128 bytes
    static constexpr int NCHUNK = D / CHUNK_COLS;
    static constexpr int TILE_BYTES = CHUNK_BYTES * NCHUNK;
    static constexpr int STAGES = (D == 128 && !F8) ? (DEC ? 6 : 4) : 8;
    // Q tiles of Q_BUFS units: with two, the producer loads the next unit's Q while the
    // current unit still computes (where shared memory has room for it).
    static constexpr int Q_BUFS = (D == 64 || F8) ? 2 : 1;
    // Q tiles per buffer: the unit's two query tiles, or the decode shape's one packed tile
    static constexpr int Q_SLOTS = DEC ? 1 : 2;
    static constexpr int SMEM_Q = 0;
    static constexpr int SMEM_KV = Q_BUFS * Q_SLOTS * TILE_BYTES;
    // bf16 epilogue staging (plain forward at d = 128): 32 rows x 128 bytes per softmax
    // warp, so that O leaves in whole 128-byte row pieces (see the epilogue)
    static constexpr bool STAGE_O = !DEC && D == 128;
    static constexpr int STG_BYTES = STAGE_O ? 8 * 32 * 128 : 0;
    static constexpr int SMEM_STG = SMEM_KV + STAGES * TILE_BYTES;
    // decode with both tiles on one split: tile 1's per-row factors for tile 0's merge,
    // [2][32] floats (1 / sum of rounded P, and the LSE); its O stays in tensor memory
    static constexpr int SMEM_XCHG = SMEM_STG + STG_BYTES;
    static constexpr int XCHG_BYTES = DEC ? 2 * 32 * 4 : 0;
    static constexpr int SMEM_BAR = SMEM_XCHG + XCHG_BYTES;
    // barrier indices
    static constexpr int B_QFULL = 0;                        // 2 * Q_BUFS: (buffer, tile)
    static constexpr int B_QEMPTY = 2 * Q_BUFS;              // Q_BUFS
    static constexpr int B_KVFULL = 3 * Q_BUFS;              // STAGES
    static constexpr int B_KVEMPTY = B_KVFULL + STAGES;      // STAGES
    static constexpr int B_SFULL = B_KVEMPTY + STAGES;       // 2
    static constexpr int B_PFULL = B_SFULL + 2;     // 4: (tile, half of P)
    static constexpr int B_OFULL = B_PFULL + 4;     // 2
    static constexpr int B_SFREE = B_OFULL + 2;     // 2: softmax has read S_t (separate-P mode)
    static constexpr int B_PVDONE = B_SFREE + 2;    // 2: a P.V product of tile t completed
    static constexpr int B_XFULL = B_PVDONE + 2;    // 1: decode, tile 1's factors are in shared memory
    static constexpr int B_XEMPTY = B_XFULL + 1;    // 1: decode, tile 0 has read them and O_1
    static constexpr int B_DRAIN = B_XEMPTY + 1;    // 1
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int SMEM_CTL = SMEM_BAR + NUM_BARS * 8;
    static constexpr int SMEM_TOTAL = SMEM_CTL + 16;
    static constexpr int SMEM_ALLOC = SMEM_TOTAL + 1024;  // room to align to 1024 bytes
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
    // Separate-P mode: when two S blocks, two O blocks and two 64-column P blocks fit in
    // tensor memory (d = 64), P gets columns of its own. S_t(j+1) can then be computed as
    // soon as the softmax warps have read S_t(j), while they are still turning it into
    // P. Otherwise (d = 128) P overwrites the first half of its S block, and S_t(j+1)
    // must wait until the P.V product of tile j has read P.
    static constexpr bool SEP_P = !F8 && (256 + 2 * D + 2 * 64) <= (int)TMEM_COLS;
    // tensor-memory columns that hold one tile's P: 128 keys, 2 (bf16) or 4 (e4m3) per column
    static constexpr int P_COLS = BN * ELEM / 4;
    static constexpr uint32_t COL_P0 = SEP_P ? 256 + 2 * D : COL_S0;
    static constexpr uint32_t COL_P1 = SEP_P ? 256 + 2 * D + 64 : COL_S1;
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * D <= (int)TMEM_COLS, "tensor memory budget");
};

struct Ctl {
    uint32_t tmem_base;
    uint32_t abort;
};

// ------------------------------------------------------------------ bounded waits
__device__ __forceinline__ void raise_timeout(volatile uint32_t *abort_flag) {
    *abort_flag = 1u;
    atomicOr(&g_status, STATUS_TIMEOUT);
}

// single-thread wait; false once the limit passes or another role gave up
__device__ bool wait_one(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                         unsigned long long limit) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait_sleep(bar, parity, WAIT_SLEEP_NS)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > limit) {
            raise_timeout(abort_flag);
            return false;
        }
    }
}

// whole-warp wait; every lane returns the same value
__device__ bool wait_warp(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                          unsigned long long limit) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    // fast path: the phase has usually completed already
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
    while (true) {
        const bool ok = ptx::mbar_try_wait_sleep(bar, parity, WAIT_SLEEP_NS);
        if (__all_sync(0xffffffffu, ok)) return true;
        int give_up = 0;
        if (lane == 0) {
            const uint64_t now = ptx::globaltimer_ns();
            if (t0 == 0) t0 = now;
            give_up = (*abort_flag != 0u) || (now - t0 > limit);
        }
        give_up = __shfl_sync(0xffffffffu, give_up, 0);
        if (give_up) {
            if (lane == 0) raise_timeout(abort_flag);
            return false;
        }
    }
}

// wait for copies in flight on the way out of an aborted run (bounded, no flag)
__device__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > limit) return;
    }
}

// ------------------------------------------------------------------ work units
// Unit u -> (batch b, query head hq, pair of query tiles). Pairs are visited from
// the last (the most KV tiles under a causal mask) to the first, so the heavy
// units start first; consecutive units share the pair index and walk hq fastest,
// so the G query heads that read one KV head run side by side.
struct Unit {
    int b, hq, hkv, pair;
};

__device__ __forceinline__ Unit decode_unit(int u, const Params &p) {
    const int pr = fdiv(u, p.div_bh);
    const int bh = u - pr * (p.B * p.Hq);
    Unit w;
    w.pair = p.n_pairs - 1 - pr;
    w.b = fdiv(bh, p.div_hq);
    w.hq = bh - w.b * p.Hq;
    w.hkv = fdiv(w.hq, p.div_group);
    return w;
}

// The k-th unit of this CTA: rounds of gridDim.x units go to the CTAs in alternating
// directions (0..G-1, then G-1..0), so a CTA that drew a heavy unit in one round draws
// a light one in the next. Units are numbered heaviest first.
__device__ __forceinline__ int snake_unit(int k) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// KV tile range [lo, hi) that query tile starting at row q0 must visit; empty when
// the tile lies past the end of the sequence. Tiles outside the range are fully
// masked and never loaded.
// Valid length of batch b: key_len[b] clamped to [0, N], or N without padding.
__device__ __forceinline__ int valid_len(const Params &p, int b) {
    if (!p.key_len) return p.N;
    if (!ATTN_CHECK(b >= 0 && b < p.B, 8u)) return 0;
    return min(max(__ldg(p.key_len + b), 0), p.N);
}

// Row i of a batch with valid length L sees the keys j of one interval:
//   i >= L (a padded row): none
//   otherwise j <= min(L - 1, causal ? i : N - 1, symmetric window ? i + W - 1 : N - 1)
//   and       j >= (window ? i - W + 1 : 0)
// Both ends grow with i, so the KV tiles a query tile needs are those between the
// first row's lower end and the last valid row's upper end; tiles outside are fully
// masked and never loaded. An empty range means every row of the tile is padding.
__device__ __forceinline__ void tile_range(const Params &p, int q0, int L, int &lo, int &hi) {
    lo = 0;
    hi = 0;
    const int rows_end = min(L, q0 + BM);  // valid rows are [q0, rows_end)
    if (q0 >= rows_end) return;
    const int r_last = rows_end - 1;
    int last_key = L - 1;
    if (p.causal) last_key = min(last_key, r_last);
    if (p.sym) last_key = min(last_key, r_last + p.window - 1);
    hi = last_key / BN + 1;
    if (p.window > 0) {
        const int first = q0 - p.window + 1;  // first visible key of row q0
        lo = first > 0 ? first / BN : 0;
    }
}

// a (query tile, key tile) block needs element masking when it crosses the end of
// the sequence, the causal diagonal or the window edge
// (rows at positions pos_first .. pos_last; padded: some rows are padding)
__device__ __forceinline__ bool block_needs_mask(const Params &p, int pos_first, int pos_last,
                                                 int kv0, int L, bool padded) {
    if (kv0 + BN > L) return true;                                      // keys past the valid end
    if (padded) return true;                                            // padded query rows
    if (p.causal && kv0 + BN - 1 > pos_first) return true;              // the diagonal
    if (p.window > 0 && pos_last - kv0 >= p.window) return true;        // the window's lower edge
    if (p.sym && kv0 + BN - 1 > pos_first + p.window - 1) return true;  // the upper edge
    return false;
}

// query/output rows of one split in the decode shape: rows per z index x z indices
__device__ __forceinline__ size_t rows_per_split(const Params &p) {
    return static_cast<size_t>(p.N) * static_cast<size_t>(p.B) * static_cast<size_t>(p.Hkv);
}

// What a work unit covers: the tensor-map z index of its query/output rows and of its
// keys/values, the first row of its first query tile (the second starts BM rows
// later), the key tiles [lo_t, hi_t) each query tile visits, and the valid key length.
struct UnitInfo {
    int zq, zkv, q0a, L, split;
    int lo0, hi0, lo1, hi1;
};

template <bool DEC>
__device__ __forceinline__ UnitInfo unit_info(int u, const Params &p) {
    UnitInfo ui;
    if constexpr (!DEC) {
        const Unit w = decode_unit(u, p);
        ui.zq = w.b * p.Hq + w.hq;
        ui.zkv = w.b * p.Hkv + w.hkv;
        ui.q0a = 2 * w.pair * BM;
        ui.L = valid_len(p, w.b);
        ui.split = 0;
        tile_range(p, ui.q0a, ui.L, ui.lo0, ui.hi0);
        tile_range(p, ui.q0a + BM, ui.L, ui.lo1, ui.hi1);
    } else {
        // one query tile holding the G * Nq rows that read KV head zkv; the split takes
        // a contiguous share of the key tiles the rows can see
        const int bhkv = fdiv(u, p.div_splits);
        ui.split = u - bhkv * p.splits;
        ui.zq = ui.zkv = bhkv;
        ui.q0a = 0;
        ui.L = p.Nk;
        ui.lo0 = p.split_lo + ui.split * p.split_len;
        ui.hi0 = min(ui.lo0 + p.split_len, p.split_hi);
        if (ui.hi0 <= ui.lo0) ui.lo0 = ui.hi0 = 0;  // nothing left for this split
        ui.lo1 = ui.hi1 = 0;
        // both tiles on the split: tile 0 from the first key tile, tile 1 from the second,
        // each taking every other tile up to hi
        if (p.dec2 && ui.hi0 > ui.lo0 + 1) {
            ui.lo1 = ui.lo0 + 1;
            ui.hi1 = ui.hi0;
        }
    }
    return ui;
}

// ------------------------------------------------------------------ kernel
template <int D, bool DEC, bool F8>
__global__ void attn_fwd_kernel(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                                const __grid_constant__ CUtensorMap, const Params);

// Launches the forward kernel as a programmatic dependent of the previous kernel on the
// stream (see the kernel's prologue).
template <int D, bool DEC, bool F8>
cudaError_t launch_fwd_kernel(int grid, size_t smem, cudaStream_t stream, const CUtensorMap &mq,
                              const CUtensorMap &mk, const CUtensorMap &mv, const Params &p) {
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(NUM_THREADS);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    lc.attrs = la;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, attn_fwd_kernel<D, DEC, F8>, mq, mk, mv, p);
}

template <int D, bool DEC, bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const Params p) {
    using C = Cfg<D, F8, DEC>;
    static_assert(!F8 || (D == 128 && !DEC), "e4m3 operands: d = 128, plain forward");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + C::SMEM_CTL);
    auto bar = [&](int i) -> uint32_t { return sb + C::SMEM_BAR + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // decode with splits: the merge kernel that follows may be scheduled now (it waits for
    // this grid's completion before reading anything)
    if constexpr (DEC) {
        if (p.splits > 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }

    if (threadIdx.x == 0) {
        for (int b = 0; b < C::Q_BUFS; ++b) {
            ptx::mbar_init(bar(C::B_QFULL + 2 * b + 0), 1);
            ptx::mbar_init(bar(C::B_QFULL + 2 * b + 1), 1);
            ptx::mbar_init(bar(C::B_QEMPTY + b), 1);
        }
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(bar(C::B_KVFULL + s), 1);
            ptx::mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar(C::B_SFULL + t), 1);
            ptx::mbar_init(bar(C::B_PFULL + 2 * t + 0), 4);  // one arrival per softmax warp
            ptx::mbar_init(bar(C::B_PFULL + 2 * t + 1), 4);
            ptx::mbar_init(bar(C::B_OFULL + t), 1);
            ptx::mbar_init(bar(C::B_SFREE + t), 4);
            ptx::mbar_init(bar(C::B_PVDONE + t), 1);
        }
        ptx::mbar_init(bar(C::B_XFULL), 1);
        ptx::mbar_init(bar(C::B_XEMPTY), 1);
        ptx::mbar_init(bar(C::B_DRAIN), 1);
        ctl->abort = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == WARP_TMA && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == WARP_MMA) {
        ptx::tmem_alloc(sb + C::SMEM_CTL, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile uint32_t *abort_flag = &ctl->abort;
    const unsigned long long limit = p.timeout_ns;
    // Programmatic dependent launch: the prologue above may overlap the end of the kernel
    // before this one on the stream (another attention call, say); every memory access
    // of the pass comes after this wait for it to complete. A dependent launched after
    // this kernel may be scheduled from now on; it waits likewise.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (!DEC) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp >= 8) {
        ptx::setmaxnreg_dec<PRODUCER_REGS>();
        if (warp == WARP_TMA) {
            // ============================================================ TMA producer
            // All 32 lanes run this loop with identical values; each copy is issued by one
            // elected lane.
            uint32_t kv_it = 0, q_it = 0;
            bool ok = true;
            for (int k = 0, u = snake_unit(0); ok && u < p.num_units; u = snake_unit(++k)) {
                const UnitInfo ui = unit_info<DEC>(u, p);
                const int q0a = ui.q0a, q0b = q0a + BM;
                const int lo0 = ui.lo0, hi0 = ui.hi0, lo1 = ui.lo1, hi1 = ui.hi1;
                // a first tile without visible keys has only padded rows (or an empty
                // split), and so has the second: nothing to load (the softmax warps write
                // the zero output)
                if (hi0 <= lo0) continue;
                const bool has1 = hi1 > lo1;
                const int lo = has1 ? min(lo0, lo1) : lo0;
                const int hi = has1 ? max(hi0, hi1) : hi0;
                const int zq = ui.zq;
                const int zkv = ui.zkv;
                // Q buffer of this unit; its previous contents (the unit Q_BUFS units
                // back) are free once that unit's last S product has completed
                const uint32_t qb = q_it % C::Q_BUFS, qph = (q_it / C::Q_BUFS) & 1u;
                ok = wait_warp(bar(C::B_QEMPTY + qb), qph ^ 1u, abort_flag, limit);
                if (!ok) break;
                ++q_it;
                const uint32_t qdst = sb + C::SMEM_Q + qb * C::Q_SLOTS * C::TILE_BYTES;
                // debug build: the Q buffer and the tensor-map z index of the unit's rows
                if (!ATTN_CHECK(qb < static_cast<uint32_t>(C::Q_BUFS) && zq >= 0 &&
                                    zq < (DEC ? p.B * p.Hkv : p.B * p.Hq) && q0a >= 0 && q0a < p.N,
                                1u))
                    continue;
                ptx::mbar_arrive_expect_tx_elect(bar(C::B_QFULL + 2 * qb + 0), C::TILE_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCHUNK; ++c)
                    ptx::tma_load_3d_elect(qdst + c * C::CHUNK_BYTES, &tm_q, bar(C::B_QFULL + 2 * qb + 0),
                                           c * C::CHUNK_COLS, q0a, zq);
                if (has1 && !DEC) {
                    ptx::mbar_arrive_expect_tx_elect(bar(C::B_QFULL + 2 * qb + 1), C::TILE_BYTES);
#pragma unroll
                    for (int c = 0; c < C::NCHUNK; ++c)
                        ptx::tma_load_3d_elect(qdst + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_q,
                                               bar(C::B_QFULL + 2 * qb + 1), c * C::CHUNK_COLS, q0b, zq);
                } else if (lane == 0) {
                    // no second tile (or the decode shape, whose second tile reads the first
                    // tile's Q): complete the phase anyway, so that both barriers of a buffer
                    // always advance together
                    ptx::mbar_arrive(bar(C::B_QFULL + 2 * qb + 1));
                }
                // K (kv = 0) or V (kv = 1) of key tile j into the next ring stage
                auto load_kv = [&](int j, int kv) -> bool {
                    const uint32_t st = kv_it % C::STAGES;
                    const uint32_t ph = ((kv_it / C::STAGES) & 1u) ^ 1u;
                    if (!wait_warp(bar(C::B_KVEMPTY + st), ph, abort_flag, limit)) return false;
                    ++kv_it;
                    // debug build: the ring stage, the KV head and the key tile
                    if (!ATTN_CHECK(st < static_cast<uint32_t>(C::STAGES) && zkv >= 0 && zkv < p.B * p.Hkv && j >= 0 &&
                                        j * BN < p.Nk,
                                    2u))
                        return true;
                    ptx::mbar_arrive_expect_tx_elect(bar(C::B_KVFULL + st), C::TILE_BYTES);
                    const CUtensorMap *m = kv ? &tm_v : &tm_k;
#pragma unroll
                    for (int c = 0; c < C::NCHUNK; ++c)
                        ptx::tma_load_3d_elect(sb + C::SMEM_KV + st * C::TILE_BYTES + c * C::CHUNK_BYTES, m,
                                               bar(C::B_KVFULL + st), c * C::CHUNK_COLS, j * BN, zkv);
                    return true;
                };
                if (DEC && p.dec2) {
                    // both tiles on the split: key tiles in pairs, K K V V, in the order the
                    // two tiles' products read them
                    for (int j = lo0; ok && j < hi0; j += 2) {
                        const bool two = j + 1 < hi0;
                        ok = load_kv(j, 0);
                        if (ok && two) ok = load_kv(j + 1, 0);
                        if (ok) ok = load_kv(j, 1);
                        if (ok && two) ok = load_kv(j + 1, 1);
                    }
                } else {
                    for (int j = lo; ok && j < hi; ++j) {
                        ok = load_kv(j, 0);  // K_j, then V_j
                        if (ok) ok = load_kv(j, 1);
                    }
                }
            }
            if (!ok) {
                // let every copy this warp issued land before the CTA exits
                for (uint32_t st = 0; st < static_cast<uint32_t>(C::STAGES); ++st) {
                    if (kv_it <= st) continue;
                    const uint32_t last = (kv_it - 1u - st) / C::STAGES * C::STAGES + st;
                    drain_wait(bar(C::B_KVFULL + st), (last / C::STAGES) & 1u, 100000000ull);
                }
                for (uint32_t b = 0; b < static_cast<uint32_t>(C::Q_BUFS); ++b) {
                    const uint32_t n_b = (q_it + C::Q_BUFS - 1u - b) / C::Q_BUFS;  // loads into buffer b
                    if (n_b == 0) continue;
                    drain_wait(bar(C::B_QFULL + 2 * b + 0), (n_b - 1u) & 1u, 100000000ull);
                    drain_wait(bar(C::B_QFULL + 2 * b + 1), (n_b - 1u) & 1u, 100000000ull);
                }
            }
        } else if (warp == WARP_MMA) {
            // ============================================================ MMA issuer
            // All 32 lanes run this loop with identical values (so descriptors and tensor
            // memory addresses are warp-uniform); each MMA and commit is issued by one
            // elected lane.
            constexpr uint32_t IDESC_S = F8 ? ptx::idesc_e4m3_f32(BM, BN, false) : ptx::idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t IDESC_PV = F8 ? ptx::idesc_e4m3_f32(BM, D, true) : ptx::idesc_bf16_f32(BM, D, true);
            uint32_t kv_it = 0, q_use = 0, p_use0 = 0, p_use1 = 0;
            uint32_t sf_use0 = 0, sf_use1 = 0;
            bool ok = true;

            // S_t = Q_t K^T: K-major A and B, 16 columns of d (32 bytes) per instruction.
            // The descriptors of later K steps differ only in the start-address field:
            // four steps of 32 bytes cover one 128-byte swizzled slab, and each slab of
            // four is issued from one asm statement (one elected lane, one predicate set-up;
            // the MMA warp's instruction count per MMA bounds how fast it feeds the
            // tensor core).
            auto issue_s = [&](uint32_t qa, uint32_t col_s, uint32_t kslot) {
                // debug build: the K stage, the Q tiles inside their region, S inside tensor memory
                if (!ATTN_CHECK(kslot < static_cast<uint32_t>(C::STAGES) && qa >= sb + C::SMEM_Q &&
                                    qa + C::TILE_BYTES <= sb + C::SMEM_KV && col_s + BN <= TMEM_COLS,
                                3u))
                    return;
                const uint64_t qd = ptx::sdesc_sw128(qa, 16, 1024);
                const uint64_t kd = ptx::sdesc_sw128(sb + C::SMEM_KV + kslot * C::TILE_BYTES, 16, 1024);
#pragma unroll
                for (int g = 0; g < D / C::KSTEP / 4; ++g) {
                    const uint64_t off = static_cast<uint64_t>(g * C::CHUNK_BYTES) >> 4;
                    ptx::mma_ss4_elect<2, F8>(tmem + col_s, qd + off, kd + off, IDESC_S, g > 0 ? 1u : 0u);
                }
            };
            // O_t (+)= P_t V: P from tensor memory (K-major), V MN-major in shared memory.
            // The softmax warps hand P over in two halves of 64 keys each; the MMAs of
            // the first half are issued as soon as it is written, while the second half
            // is still being computed.
            auto issue_pv = [&](int t, uint32_t col_o, uint32_t col_s, uint32_t vslot,
                                bool accumulate, uint32_t parity) -> bool {
                // debug build: the V stage, O and P inside tensor memory
                const bool in_range = ATTN_CHECK(vslot < static_cast<uint32_t>(C::STAGES) &&
                                                     col_o + D <= TMEM_COLS && col_s + C::P_COLS <= TMEM_COLS,
                                                 4u);
                const uint64_t vd = ptx::sdesc_sw128(sb + C::SMEM_KV + vslot * C::TILE_BYTES,
                                                     C::CHUNK_BYTES, 1024);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    if (!wait_warp(bar(C::B_PFULL + 2 * t + h), parity, abort_flag, limit)) return false;
                    ptx::tc_fence_after();
                    if (!in_range) continue;
                    // step k16 reads 8 tensor-memory columns of P (KSTEP keys) and the KSTEP
                    // rows of V after the previous steps' KSTEP * 128 bytes; a bf16 half is
                    // four steps, issued from one asm statement
                    if constexpr (!F8) {
                        const int k0 = h * 4;
                        ptx::mma_ts4_elect<8, 128>(tmem + col_o, tmem + col_s + k0 * 8, vd + ((k0 * 16 * 128) >> 4),
                                                   IDESC_PV, (accumulate || h > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BN / C::KSTEP / 2; ++kk) {
                            const int k16 = h * (BN / C::KSTEP / 2) + kk;
                            const uint64_t vstep = vd + ((k16 * C::KSTEP * 128) >> 4);
                            ptx::mma_ts_elect_f8(tmem + col_o, tmem + col_s + k16 * 8, vstep, IDESC_PV,
                                                 (accumulate || k16 > 0) ? 1u : 0u);
                        }
                    }
                }
                return true;
            };

            for (int k = 0, u = snake_unit(0); ok && u < p.num_units; u = snake_unit(++k)) {
                const UnitInfo ui = unit_info<DEC>(u, p);
                const int lo0 = ui.lo0, hi0 = ui.hi0, lo1 = ui.lo1, hi1 = ui.hi1;
                if (hi0 <= lo0) continue;  // padding only (or an empty split): nothing to compute
                const bool has1 = hi1 > lo1;
                const int lo = has1 ? min(lo0, lo1) : lo0;
                const int hi = has1 ? max(hi0, hi1) : hi0;
                const uint32_t qb = q_use % C::Q_BUFS, qph = (q_use / C::Q_BUFS) & 1u;
                ++q_use;
                // (the decode shape's tile 1 reads tile 0's packed Q)
                const uint32_t qa0 = sb + C::SMEM_Q + qb * C::Q_SLOTS * C::TILE_BYTES;
                const uint32_t qa1 = qa0 + (C::Q_SLOTS - 1) * C::TILE_BYTES;
                ok = wait_warp(bar(C::B_QFULL + 2 * qb + 0), qph, abort_flag, limit);
                if (ok) ok = wait_warp(bar(C::B_QFULL + 2 * qb + 1), qph, abort_flag, limit);
                if (!ok) break;
                ptx::tc_fence_after();
                int prev = -1;
                uint32_t vprev = 0, vprev_ph = 0;
                if constexpr (DEC) {
                    if (p.dec2) {
                        // Decode shape, both tiles on the split's key tiles [lo0, hi0): tile 0
                        // takes lo0, lo0 + 2, .., tile 1 lo0 + 1, lo0 + 3, .., both with the
                        // one packed Q tile. The producer loads pairs of key tiles as K K V V.
                        // A step issues both tiles' S and the previous step's P.V products;
                        // every K and V tile has one reader and is released after it.
                        const int a = lo0, bnd = hi0;
                        const int n0 = (bnd - a + 1) / 2, n1 = (bnd - a) / 2;
                        const uint32_t base = kv_it;
                        kv_it += 2u * static_cast<uint32_t>(bnd - a);
                        auto kv_index = [&](int j, uint32_t kv) -> uint32_t {
                            const int r = j - a, pr = r >> 1, t = r & 1;
                            const bool two = a + 2 * pr + 1 < bnd;
                            return base + 4u * static_cast<uint32_t>(pr) +
                                   (kv ? (two ? 2u + static_cast<uint32_t>(t) : 1u) : static_cast<uint32_t>(t));
                        };
                        auto kv_wait = [&](uint32_t it) -> bool {
                            if (!wait_warp(bar(C::B_KVFULL + it % C::STAGES), (it / C::STAGES) & 1u, abort_flag, limit))
                                return false;
                            ptx::tc_fence_after();
                            return true;
                        };
                        // S_t for key tile j (tile t's n-th), then K is released
                        auto s_dec = [&](int t, int j) -> bool {
                            const uint32_t it = kv_index(j, 0);
                            if (!kv_wait(it)) return false;
                            if constexpr (C::SEP_P) {
                                uint32_t &sf = t ? sf_use1 : sf_use0;
                                if (!wait_warp(bar(C::B_SFREE + t), (sf & 1u) ^ 1u, abort_flag, limit)) return false;
                                ++sf;
                                ptx::tc_fence_after();
                            }
                            issue_s(qa0, t ? C::COL_S1 : C::COL_S0, it % C::STAGES);
                            ptx::mma_commit_elect(bar(C::B_SFULL + t));
                            ptx::mma_commit_elect(bar(C::B_KVEMPTY + it % C::STAGES));
                            return true;
                        };
                        // O_t (+)= P_t V for tile t's k-th key tile j; the last of the unit
                        // reports O_t complete, the others (separate P) that P is free again
                        auto pv_dec = [&](int t, int j, int k, bool last) -> bool {
                            const uint32_t it = kv_index(j, 1);
                            if (!kv_wait(it)) return false;
                            uint32_t &pu = t ? p_use1 : p_use0;
                            if (!issue_pv(t, t ? C::COL_O1 : C::COL_O0, t ? C::COL_P1 : C::COL_P0, it % C::STAGES, k > 0,
                                          pu & 1u))
                                return false;
                            ++pu;
                            if (last)
                                ptx::mma_commit_elect(bar(C::B_OFULL + t));
                            else if constexpr (C::SEP_P)
                                ptx::mma_commit_elect(bar(C::B_PVDONE + t));
                            ptx::mma_commit_elect(bar(C::B_KVEMPTY + it % C::STAGES));
                            return true;
                        };
                        for (int st = 0; ok && st < n0; ++st) {
                            const int j0 = a + 2 * st, j1 = j0 + 1;
                            if constexpr (C::SEP_P) {
                                ok = s_dec(0, j0);
                                if (ok && st < n1) ok = s_dec(1, j1);
                                if (ok && st > 0) ok = pv_dec(0, j0 - 2, st - 1, false);
                                if (ok && st > 0 && st - 1 < n1) ok = pv_dec(1, j1 - 2, st - 1, st == n1);
                            } else {
                                if (st > 0) ok = pv_dec(0, j0 - 2, st - 1, false);
                                if (ok) ok = s_dec(0, j0);
                                if (ok && st > 0 && st - 1 < n1) ok = pv_dec(1, j1 - 2, st - 1, st == n1);
                                if (ok && st < n1) ok = s_dec(1, j1);
                            }
                        }
                        if (!ok) break;
                        ptx::mma_commit_elect(bar(C::B_QEMPTY + qb));  // Q free once the last S is done
                        // the last products: tile 0's always; tile 1's when it has as many key
                        // tiles as tile 0 (with one fewer, its last came in the last step)
                        ok = pv_dec(0, a + 2 * (n0 - 1), n0 - 1, true);
                        if (ok && n1 > 0 && n1 == n0) ok = pv_dec(1, a + 2 * (n1 - 1) + 1, n1 - 1, true);
                        if (!ok) break;
                        continue;
                    }
                }
                if constexpr (C::SEP_P) {
                    // S_t(j) is issued as soon as the softmax warps have read S_t(j-1);
                    // then come the P.V products of key tile j-1 for both query tiles.
                    auto pv_step = [&](int pj) -> bool {
                        if (!wait_warp(bar(C::B_KVFULL + vprev), vprev_ph, abort_flag, limit)) return false;
                        ptx::tc_fence_after();
                        if (pj >= lo0 && pj < hi0) {
                            if (!issue_pv(0, C::COL_O0, C::COL_P0, vprev, pj > lo0, p_use0 & 1u)) return false;
                            ++p_use0;
                            ptx::mma_commit_elect(bar(pj == hi0 - 1 ? C::B_OFULL + 0 : C::B_PVDONE + 0));
                        }
                        if (has1 && pj >= lo1 && pj < hi1) {
                            if (!issue_pv(1, C::COL_O1, C::COL_P1, vprev, pj > lo1, p_use1 & 1u)) return false;
                            ++p_use1;
                            ptx::mma_commit_elect(bar(pj == hi1 - 1 ? C::B_OFULL + 1 : C::B_PVDONE + 1));
                        }
                        ptx::mma_commit_elect(bar(C::B_KVEMPTY + vprev));
                        return true;
                    };
                    for (int j = lo; j < hi; ++j) {
                        const uint32_t ks = kv_it % C::STAGES, kph = (kv_it / C::STAGES) & 1u;
                        ++kv_it;
                        const uint32_t vs = kv_it % C::STAGES, vph = (kv_it / C::STAGES) & 1u;
                        ++kv_it;
                        ok = wait_warp(bar(C::B_KVFULL + ks), kph, abort_flag, limit);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        if (j >= lo0 && j < hi0) {
                            ok = wait_warp(bar(C::B_SFREE + 0), (sf_use0 & 1u) ^ 1u, abort_flag, limit);
                            ++sf_use0;
                            if (!ok) break;
                            ptx::tc_fence_after();
                            issue_s(qa0, C::COL_S0, ks);
                            ptx::mma_commit_elect(bar(C::B_SFULL + 0));
                        }
                        if (has1 && j >= lo1 && j < hi1) {
                            ok = wait_warp(bar(C::B_SFREE + 1), (sf_use1 & 1u) ^ 1u, abort_flag, limit);
                            ++sf_use1;
                            if (!ok) break;
                            ptx::tc_fence_after();
                            issue_s(qa1, C::COL_S1, ks);
                            ptx::mma_commit_elect(bar(C::B_SFULL + 1));
                        }
                        ptx::mma_commit_elect(bar(C::B_KVEMPTY + ks));
                        if (prev >= 0) {
                            ok = pv_step(prev);
                            if (!ok) break;
                        }
                        prev = j;
                        vprev = vs;
                        vprev_ph = vph;
                    }
                    if (!ok) break;
                    ptx::mma_commit_elect(bar(C::B_QEMPTY + qb));  // Q tiles free once the last S is done
                    ok = pv_step(prev);
                    if (!ok) break;
                } else if (has1 && ui.lo1 == lo0 + 1 && ui.hi1 == hi0 + 1) {
                    // A sliding window: tile 1's key range is tile 0's shifted by one tile.
                    // Tile 1 runs one key tile ahead, so both tiles compute in every step
                    // (n steps instead of n + 1, with no step for one tile alone): step j
                    // does O0 += P0 V(j-1), S0 = Q0 K(j)^T, O1 += P1 V(j), S1 = Q1 K(j+1)^T.
                    // Each K/V tile is waited for right before its first use (the ring
                    // refills while the earlier products of the step run) and released
                    // after its last. The producer's order is unchanged: K, V of key tiles
                    // lo0 .. hi0.
                    const uint32_t base = kv_it;
                    kv_it += 2u * static_cast<uint32_t>(hi - lo);
                    auto kv_slot = [&](int j, uint32_t kv) {
                        return (base + 2u * static_cast<uint32_t>(j - lo0) + kv) % C::STAGES;
                    };
                    auto kv_wait = [&](int j, uint32_t kv) -> bool {
                        const uint32_t it = base + 2u * static_cast<uint32_t>(j - lo0) + kv;
                        if (!wait_warp(bar(C::B_KVFULL + it % C::STAGES), (it / C::STAGES) & 1u, abort_flag, limit))
                            return false;
                        ptx::tc_fence_after();
                        return true;
                    };
                    ok = kv_wait(lo0, 0);
                    for (int j = lo0; ok && j < hi0; ++j) {
                        if (j > lo0) {
                            if (j - 1 == lo0) ok = kv_wait(lo0, 1);  // V(lo0): tile 1 never reads it
                            if (ok) ok = issue_pv(0, C::COL_O0, C::COL_P0, kv_slot(j - 1, 1), j - 1 > lo0, p_use0 & 1u);
                            ++p_use0;
                            if (!ok) break;
                            ptx::mma_commit_elect(bar(C::B_KVEMPTY + kv_slot(j - 1, 1)));
                        }
                        issue_s(qa0, C::COL_S0, kv_slot(j, 0));
                        ptx::mma_commit_elect(bar(C::B_SFULL + 0));
                        ptx::mma_commit_elect(bar(C::B_KVEMPTY + kv_slot(j, 0)));
                        if (j > lo0) {
                            ok = kv_wait(j, 1) &&
                                 issue_pv(1, C::COL_O1, C::COL_P1, kv_slot(j, 1), j > lo0 + 1, p_use1 & 1u);
                            ++p_use1;
                            if (!ok) break;
                        }
                        ok = kv_wait(j + 1, 0);
                        if (!ok) break;
                        issue_s(qa1, C::COL_S1, kv_slot(j + 1, 0));
                        ptx::mma_commit_elect(bar(C::B_SFULL + 1));
                        if (j + 1 >= hi0) ptx::mma_commit_elect(bar(C::B_KVEMPTY + kv_slot(j + 1, 0)));
                    }
                    if (!ok) break;
                    ptx::mma_commit_elect(bar(C::B_QEMPTY + qb));  // Q tiles free once the last S is done
                    // the last products: O0 += P0 V(hi0-1), O1 += P1 V(hi0)
                    if (hi0 - 1 == lo0) ok = kv_wait(lo0, 1);
                    if (ok) ok = issue_pv(0, C::COL_O0, C::COL_P0, kv_slot(hi0 - 1, 1), hi0 - 1 > lo0, p_use0 & 1u);
                    ++p_use0;
                    if (!ok) break;
                    ptx::mma_commit_elect(bar(C::B_OFULL + 0));
                    ptx::mma_commit_elect(bar(C::B_KVEMPTY + kv_slot(hi0 - 1, 1)));
                    ok = kv_wait(hi0, 1) && issue_pv(1, C::COL_O1, C::COL_P1, kv_slot(hi0, 1), hi0 > lo0 + 1, p_use1 & 1u);
                    ++p_use1;
                    if (!ok) break;
                    ptx::mma_commit_elect(bar(C::B_OFULL + 1));
                    ptx::mma_commit_elect(bar(C::B_KVEMPTY + kv_slot(hi0, 1)));
                } else {
                    for (int j = lo; j < hi; ++j) {
                        const uint32_t ks = kv_it % C::STAGES, kph = (kv_it / C::STAGES) & 1u;
                        ++kv_it;
                        const uint32_t vs = kv_it % C::STAGES, vph = (kv_it / C::STAGES) & 1u;
                        ++kv_it;
                        ok = wait_warp(bar(C::B_KVFULL + ks), kph, abort_flag, limit);
                        if (ok && prev >= 0) ok = wait_warp(bar(C::B_KVFULL + vprev), vprev_ph, abort_flag, limit);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        // tile 0: O0 += P0(prev) V(prev), then S0 = Q0 K_j^T
                        if (prev >= lo0 && prev < hi0) {
                            ok = issue_pv(0, C::COL_O0, C::COL_P0, vprev, prev > lo0, p_use0 & 1u);
                            ++p_use0;
                            if (!ok) break;
                        }
                        if (j >= lo0 && j < hi0) {
                            issue_s(qa0, C::COL_S0, ks);
                            ptx::mma_commit_elect(bar(C::B_SFULL + 0));
                        }
                        // tile 1: the same, overlapping softmax of tile 0
                        if (has1 && prev >= lo1 && prev < hi1) {
                            ok = issue_pv(1, C::COL_O1, C::COL_P1, vprev, prev > lo1, p_use1 & 1u);
                            ++p_use1;
                            if (!ok) break;
                        }
                        if (has1 && j >= lo1 && j < hi1) {
                            issue_s(qa1, C::COL_S1, ks);
                            ptx::mma_commit_elect(bar(C::B_SFULL + 1));
                        }
                        if (prev >= 0) ptx::mma_commit_elect(bar(C::B_KVEMPTY + vprev));
                        ptx::mma_commit_elect(bar(C::B_KVEMPTY + ks));
                        prev = j;
                        vprev = vs;
                        vprev_ph = vph;
                    }
                    if (!ok) break;
                    ptx::mma_commit_elect(bar(C::B_QEMPTY + qb));  // Q tiles free once the last S is done
                    ok = wait_warp(bar(C::B_KVFULL + vprev), vprev_ph, abort_flag, limit);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    if (prev >= lo0 && prev < hi0) {
                        ok = issue_pv(0, C::COL_O0, C::COL_P0, vprev, prev > lo0, p_use0 & 1u);
                        ++p_use0;
                        if (!ok) break;
                    }
                    ptx::mma_commit_elect(bar(C::B_OFULL + 0));
                    if (has1) {
                        if (prev >= lo1 && prev < hi1) {
                            ok = issue_pv(1, C::COL_O1, C::COL_P1, vprev, prev > lo1, p_use1 & 1u);
                            ++p_use1;
                            if (!ok) break;
                        }
                        ptx::mma_commit_elect(bar(C::B_OFULL + 1));
                    }
                    ptx::mma_commit_elect(bar(C::B_KVEMPTY + vprev));
                }
            }
            // every MMA this warp issued completes before tensor memory is freed
            ptx::mma_commit_elect(bar(C::B_DRAIN));
            drain_wait(bar(C::B_DRAIN), 0u, 100000000ull);
            __syncwarp();
        }
    } else {
        ptx::setmaxnreg_inc<SOFTMAX_REGS>();
        // ============================================================ softmax + epilogue
        const int t = warp >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t t_s = tmem + lane_off + (t ? C::COL_S1 : C::COL_S0);
        const uint32_t t_o = tmem + lane_off + (t ? C::COL_O1 : C::COL_O0);
        const uint32_t t_p = tmem + lane_off + (t ? C::COL_P1 : C::COL_P0);
        // debug build: S, O and P of this tile inside tensor memory (a failure is recorded;
        // the layout is fixed at compile time)
        (void)ATTN_CHECK((t ? C::COL_S1 : C::COL_S0) + BN <= TMEM_COLS && (t ? C::COL_O1 : C::COL_O0) + D <= TMEM_COLS &&
                             (t ? C::COL_P1 : C::COL_P0) + C::P_COLS <= TMEM_COLS,
                         5u);
        // decode shape: tile row r holds query r % Nq (of head r / Nq of the group)
        int my_dec_pos = 0;
        if constexpr (DEC) my_dec_pos = p.pos_off + (row - fdiv(row, p.div_nq) * p.Nq);
        const uint32_t bar_s = bar(C::B_SFULL + t), bar_o = bar(C::B_OFULL + t);
        const uint32_t bar_sfree = bar(C::B_SFREE + t), bar_pvdone = bar(C::B_PVDONE + t);
        uint32_t pv_w = 0;
        const uint32_t bar_p0 = bar(C::B_PFULL + 2 * t), bar_p1 = bar(C::B_PFULL + 2 * t + 1);
        const float sl2 = p.sl2;
        uint32_t s_use = 0, o_use = 0, x_use = 0;
        // decode with both tiles on a split: each tile takes every other key tile
        const int jstep = (DEC && p.dec2) ? 2 : 1;
        bool ok = true;
        for (int k = 0, u = snake_unit(0); ok && u < p.num_units; u = snake_unit(++k)) {
            const UnitInfo ui = unit_info<DEC>(u, p);
            // decode: tile 1 works only when both tiles share the split, on tile 0's rows
            if (DEC && t == 1 && !p.dec2) continue;
            const int q0 = ui.q0a + (DEC ? 0 : t * BM);
            if (q0 >= p.N) continue;  // no rows in this tile
            const int lo = t ? ui.lo1 : ui.lo0, hi = t ? ui.hi1 : ui.hi0;
            const int L = ui.L;
            const bool empty = hi <= lo;  // all rows padded (or an empty split): zero output
            const int qi = q0 + row;
            // this row's position in the sequence, and whether it is a real query row
            const int pos = DEC ? my_dec_pos : qi;
            const bool row_live = DEC ? true : (qi < L);
            // positions of the tile's first and last rows, for the edge-tile test
            const int pos_first = DEC ? p.pos_off : q0;
            const int pos_last = DEC ? p.Nk - 1 : q0 + BM - 1;
            const bool padded_rows = DEC ? false : (L < p.N && q0 + BM > L);
            // e4m3 operands: S carries the factor q_scale x k_scale of its two blocks, and
            // the V block scales are folded into P relative to the head's largest one
            // (P' = P x v_scale_j / v_max <= 256), so that O = v_max x sum P' V8 / sum P
            float q_sc = 1.f, v_max = 1.f;
            if constexpr (F8) {
                // debug build: the query block's scale lies inside the scale array
                if (ATTN_CHECK(ui.zq < p.B * p.Hq && q0 / BM < p.n_kv, 9u))
                    q_sc = __ldg(p.q_scale + static_cast<size_t>(ui.zq) * p.n_kv + (q0 / BM));
                float vm = 0.f;
                for (int jj = lane; jj < p.n_kv; jj += 32)
                    vm = fmaxf(vm, __ldg(p.v_scale + static_cast<size_t>(ui.zkv) * p.n_kv + jj));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                v_max = vm;
            }
            float m_run = -INFINITY;  // running max of scale*s*log2(e)
            float l_run = 0.f;        // running sum of 2^(x - m_run), for the LSE
            float r_run = 0.f;        // running sum of bf16(2^(x - m_run)), for normalising O
            for (int j = lo; j < hi; j += jstep) {
                ok = wait_warp(bar_s, s_use & 1u, abort_flag, limit);
                ++s_use;
                if (!ok) break;
                ptx::tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) ptx::tmem_ld32(t_s + 32 * c, sr[c]);
                ptx::tmem_wait_ld();
                if constexpr (C::SEP_P) {
                    // S_t is in registers: the tensor core may overwrite it with S_t(j+1)
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar_sfree);
                }
                const int kv0 = j * BN;
                if (block_needs_mask(p, pos_first, pos_last, kv0, L, padded_rows)) {
                    // The keys row qi sees in this tile form one interval of columns
                    // [c_lo, c_hi]: c_hi from the sequence end and the causal diagonal,
                    // c_lo from the window. One unsigned compare per element against the
                    // column index (a compile-time constant) keeps this rarely run block
                    // small.
                    int c_hi = L - 1;
                    if (p.causal) c_hi = min(c_hi, pos);
                    if (p.sym) c_hi = min(c_hi, pos + p.window - 1);
                    c_hi -= kv0;
                    const int c_lo = p.window > 0 ? max(pos - p.window + 1 - kv0, 0) : 0;
                    // an empty interval (or a padded row) becomes c_lo = -1, span = 0:
                    // every offset is then > 0
                    const bool none = c_hi < c_lo || !row_live;
                    const uint32_t span = none ? 0u : static_cast<uint32_t>(c_hi - c_lo);
                    const uint32_t base = none ? 0xFFFFFFFFu : static_cast<uint32_t>(c_lo);
                    // The warp's 32 rows decide each 32-column chunk together: a chunk that
                    // lies inside every row's interval is skipped, and only the others are
                    // compared element by element (on a diagonal tile, warp w skips the w
                    // chunks left of the diagonal; at a ragged sequence end, the chunks
                    // before it). An empty row counts as the interval [BN, -1]. The skip
                    // test needs c_lo >= 0 (the max above): a negative lower end would make
                    // lo_max understate where some row's interval starts. (A third, all
                    // -inf branch for chunks outside every interval made the compiler
                    // spill the S registers.)
                    // A row past the tensor's end (q0 + row >= N: its output is never
                    // stored) takes no part in the decision: it counts as the whole tile.
                    // Rows inside N past a batch's key length must still come out as O = 0.
                    const bool unstored = (DEC ? row : qi) >= p.N;
                    const int lo_r = unstored ? 0 : (none ? BN : c_lo), hi_r = unstored ? BN - 1 : (none ? -1 : c_hi);
                    const int lo_max = __reduce_max_sync(0xffffffffu, lo_r);
                    const int hi_min = __reduce_min_sync(0xffffffffu, hi_r);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (!(lo_max <= 32 * c && hi_min >= 32 * c + 31)) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                sr[c][e] = ptx::mask_above(sr[c][e], static_cast<uint32_t>(c * 32 + e) - base, span);
                        }
                    }
                }
                // row maximum: four independent chains of three-input max
                float mxc[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float a = __uint_as_float(sr[c][0]);
#pragma unroll
                    for (int e = 1; e < 31; e += 2)
                        a = ptx::fmax3(a, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
                    mxc[c] = fmaxf(a, __uint_as_float(sr[c][31]));
                }
                float c_tile = sl2, log_ratio = 0.f, inv_ratio = 1.f;
                if constexpr (F8) {
                    const size_t kb = static_cast<size_t>(ui.zkv) * p.n_kv + j;
                    c_tile = sl2 * q_sc * __ldg(p.k_scale + kb);
                    const float ratio = __ldg(p.v_scale + kb) / v_max;
                    log_ratio = ptx::lg2(ratio);
                    inv_ratio = 1.f / ratio;
                }
                const float mx = ptx::fmax3(mxc[0], mxc[1], fmaxf(mxc[2], mxc[3])) * c_tile;
                float m_new = m_run;
                if (mx > m_run + RESCALE_THRESHOLD) m_new = mx;
                const float alpha = (m_new == m_run) ? 1.f : ptx::ex2(m_run - m_new);
                m_run = m_new;
                const float mref = (m_run == -INFINITY) ? 0.f : m_run;

                // O <- alpha * O, only when some row of this warp raised its maximum; the
                // first KV tile needs none (its PV product overwrites O). The previous PV
                // product must have completed: with P aliasing S, the S commit this warp
                // waited for follows it; with separate P, wait for it here (this also
                // frees the P block for this tile's P).
                if constexpr (C::SEP_P) {
                    if (j > lo) {
                        ok = wait_warp(bar_pvdone, pv_w & 1u, abort_flag, limit);
                        ++pv_w;
                        if (!ok) break;
                        ptx::tc_fence_after();
                    }
                }
                if (j > lo && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld32(t_o + 32 * c, r);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        ptx::tmem_st32(t_o + 32 * c, r);
                    }
                }

                // P = 2^(x - m) as bf16 over the first half of S, handed to the MMA warp in
                // two halves of 64 keys. Two row sums: the exact one (for the LSE) and the
                // sum of the ROUNDED P, by which O is normalised: O is then an exact convex
                // combination of V rows under the weights the tensor core actually used,
                // so the rounding of a dominant weight cancels instead of showing in O.
                const float2 sl2x2 = make_float2(c_tile, c_tile);
                const float2 negm = make_float2(log_ratio - mref, log_ratio - mref);
                float2 le0 = make_float2(0.f, 0.f), le1 = make_float2(0.f, 0.f);
                float lr0 = 0.f, lr1 = 0.f, lr2 = 0.f, lr3 = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int c = 2 * h; c < 2 * h + 2; ++c) {
                        if constexpr (F8) {
                            // four e4m3 codes per tensor-memory column (key k in byte k % 4)
                            uint32_t pk[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float2 x01 = make_float2(__uint_as_float(sr[c][4 * e]),
                                                               __uint_as_float(sr[c][4 * e + 1]));
                                const float2 x23 = make_float2(__uint_as_float(sr[c][4 * e + 2]),
                                                               __uint_as_float(sr[c][4 * e + 3]));
                                const float2 a01 = __ffma2_rn(x01, sl2x2, negm);
                                const float2 a23 = __ffma2_rn(x23, sl2x2, negm);
                                const float2 p01 = make_float2(ptx::ex2(a01.x), ptx::ex2(a01.y));
                                const float2 p23 = make_float2(ptx::ex2(a23.x), ptx::ex2(a23.y));
                                pk[e] = ptx::pack_e4m3x4(p01.x, p01.y, p23.x, p23.y);
                                le0 = __fadd2_rn(le0, p01);
                                le1 = __fadd2_rn(le1, p23);
                                if (e & 1)
                                    ptx::add_e4m3x4(lr2, lr3, pk[e]);
                                else
                                    ptx::add_e4m3x4(lr0, lr1, pk[e]);
                            }
                            ptx::tmem_st8(t_p + 8 * c, pk);
                        } else {
                            uint32_t pk[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 x = make_float2(__uint_as_float(sr[c][2 * e]),
                                                             __uint_as_float(sr[c][2 * e + 1]));
                                const float2 a = __ffma2_rn(x, sl2x2, negm);
                                const float2 pe = make_float2(ptx::ex2(a.x), ptx::ex2(a.y));
                                pk[e] = ptx::pack_bf16x2(pe.x, pe.y);
                                if (e & 1) {
                                    le1 = __fadd2_rn(le1, pe);
                                    ptx::add_bf16x2_halves(lr2, lr3, pk[e]);
                                } else {
                                    le0 = __fadd2_rn(le0, pe);
                                    ptx::add_bf16x2_halves(lr0, lr1, pk[e]);
                                }
                            }
                            ptx::tmem_st16(t_p + 16 * c, pk);
                        }
                    }
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(h ? bar_p1 : bar_p0);
                }
                // (with e4m3 operands the sums are of P' = P x ratio: back to P's units)
                l_run = l_run * alpha + ((le0.x + le0.y) + (le1.x + le1.y)) * inv_ratio;
                r_run = r_run * alpha + ((lr0 + lr1) + (lr2 + lr3)) * inv_ratio;
            }
            if (!ok) break;
            if (!empty) {
                ok = wait_warp(bar_o, o_use & 1u, abort_flag, limit);
                ++o_use;
                if (!ok) break;
                ptx::tc_fence_after();
            }
            // epilogue: O / (sum of rounded P) and the natural-log LSE
            const float inv_l = r_run > 0.f ? v_max / r_run : 0.f;
            const size_t ridx = static_cast<size_t>(ui.zq) * static_cast<size_t>(p.N) +
                                static_cast<size_t>(qi);
            const float lse_nat = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
            if constexpr (DEC) {
                if (p.dec2) {
                    // Tile 1 hands tile 0 its rows' factors (1 / sum of rounded P, and the
                    // LSE) through shared memory. Its O stays in tensor memory, where tile 0
                    // reads it: the packed rows (at most 32) are the first warp's in both
                    // tiles, so the same lanes hold them. Tile 0 merges the two by
                    // log-sum-exp, as the split combine does, and writes the result. Tile 1's
                    // first P.V product of its next unit overwrites O_1, so its warp goes on
                    // only once tile 0 has read it.
                    if (quad != 0) continue;
                    float *xs = reinterpret_cast<float *>(smem + C::SMEM_XCHG);
                    if (t == 1) {
                        xs[lane] = inv_l;
                        xs[32 + lane] = lse_nat;
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(C::B_XFULL));
                        ok = wait_warp(bar(C::B_XEMPTY), x_use & 1u, abort_flag, limit);
                        ++x_use;
                        if (!ok) break;
                        continue;
                    }
                    ok = wait_warp(bar(C::B_XFULL), x_use & 1u, abort_flag, limit);
                    ++x_use;
                    if (!ok) break;
                    // tile 1 saw its last P.V product complete before it signalled
                    ptx::tc_fence_after();
                    const float inv_l1 = xs[lane], lse1 = xs[32 + lane];
                    const bool empty1 = ui.hi1 <= ui.lo1;
                    const uint32_t t_o1 = tmem + lane_off + C::COL_O1;
                    const float mx2 = fmaxf(lse_nat, lse1);
                    float w0 = 0.f, w1 = 0.f, lse_m = -INFINITY;
                    if (mx2 != -INFINITY) {
                        const float e0 = expf(lse_nat - mx2), e1 = expf(lse1 - mx2);
                        w0 = e0 / (e0 + e1);
                        w1 = e1 / (e0 + e1);
                        lse_m = mx2 + logf(e0 + e1);
                    }
                    const size_t rows_out = static_cast<size_t>(p.B * p.Hkv) * static_cast<size_t>(p.N) *
                                            static_cast<size_t>(p.splits > 1 ? p.splits : 1);
                    const size_t prow = p.splits > 1 ? static_cast<size_t>(ui.split) * rows_per_split(p) + ridx : ridx;
                    const bool store_row = qi < p.N && ATTN_CHECK(prow < rows_out, 10u);
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32], r1[32];
                        if (!empty) ptx::tmem_ld32(t_o + 32 * c, r);
                        if (!empty1) ptx::tmem_ld32(t_o1 + 32 * c, r1);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            if (empty) r[e] = 0u;
                            if (empty1) r1[e] = 0u;
                        }
                        float v[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float x1 = __uint_as_float(r1[e]) * inv_l1;
                            v[e] = __uint_as_float(r[e]) * inv_l * w0 + x1 * w1;
                        }
                        if (!store_row) continue;
                        if (p.splits > 1) {
                            float4 *dst = reinterpret_cast<float4 *>(p.o_part + prow * D) + 8 * c;
#pragma unroll
                            for (int g = 0; g < 8; ++g)
                                dst[g] = make_float4(v[4 * g + 0], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(p.o + ridx * D) + 4 * c;
#pragma unroll
                            for (int g = 0; g < 4; ++g)
                                dst[g] = make_uint4(ptx::pack_bf16x2(v[8 * g + 0], v[8 * g + 1]),
                                                    ptx::pack_bf16x2(v[8 * g + 2], v[8 * g + 3]),
                                                    ptx::pack_bf16x2(v[8 * g + 4], v[8 * g + 5]),
                                                    ptx::pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
                        }
                    }
                    if (store_row) (p.splits > 1 ? p.lse_part : p.lse)[prow] = lse_m;
                    // O_1 has been read (and the factors): tile 1 may go on
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(C::B_XEMPTY));
                    continue;
                }
            }
            // fp32 rows: the split results of the decode shape (merged later by the
            // combine kernel), or the plain forward's O when fp32 output was asked for.
            // The tensor-memory loads are warp-collective: every lane takes them, and
            // only rows of the tile store.
            float *o32_row = nullptr;
            float *lse32 = p.lse;
            size_t lse_idx = ridx;
            if constexpr (DEC) {
                if (p.splits > 1) {
                    const size_t prow = static_cast<size_t>(ui.split) * rows_per_split(p) + ridx;
                    o32_row = p.o_part + prow * D;
                    lse32 = p.lse_part;
                    lse_idx = prow;
                }
            } else {
                if (p.o32) o32_row = p.o32 + ridx * D;
            }
            // debug build: the row lies inside the output (or the split results) it is written to
            const size_t rows_out = static_cast<size_t>(DEC ? p.B * p.Hkv : p.B * p.Hq) * static_cast<size_t>(p.N) *
                                    static_cast<size_t>(DEC && p.splits > 1 ? p.splits : 1);
            if (o32_row) {
                const bool store_row = qi < p.N && ATTN_CHECK(lse_idx < rows_out, 6u);
                float4 *dst = reinterpret_cast<float4 *>(o32_row);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    if (!empty) {
                        ptx::tmem_ld32(t_o + 32 * c, r);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = 0u;
                    }
                    if (store_row) {
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            dst[c * 8 + g] = make_float4(__uint_as_float(r[4 * g + 0]) * inv_l,
                                                         __uint_as_float(r[4 * g + 1]) * inv_l,
                                                         __uint_as_float(r[4 * g + 2]) * inv_l,
                                                         __uint_as_float(r[4 * g + 3]) * inv_l);
                    }
                }
                if (store_row) lse32[lse_idx] = lse_nat;
                continue;
            }
            // O / (sum of rounded P) -> bf16, from tensor memory straight to global memory:
            // each thread writes its own row (2d contiguous bytes; rows past N are
            // skipped). The tensor-memory loads are warp-collective, so every lane takes
            // them.
            const bool store_row = qi < p.N && ATTN_CHECK(ridx < rows_out, 7u);
            if constexpr (C::STAGE_O) {
                // Each thread's row in 16-byte pieces would make every store instruction
                // touch 32 rows (32 partial sectors). Instead, for each 64-column (128-byte)
                // piece of the rows, the warp's 32 rows go through its own staging block
                // (16-byte units of row r at unit u ^ (r % 8), conflict-free both ways) and
                // leave with 8 lanes per row: 4 whole 128-byte lines per instruction. (At
                // d = 64, where a row is one such piece, the direct stores are as fast.)
                const uint32_t stg = sb + C::SMEM_STG + static_cast<uint32_t>(warp) * 32u * 128u;
                const uint32_t sw = static_cast<uint32_t>(lane & 7);
                // the row this lane stores in round k: warp row (lane / 8) + 4k
                const int rr0 = lane >> 3, part = lane & 7;
                const size_t rbase = static_cast<size_t>(ui.zq) * static_cast<size_t>(p.N) +
                                     static_cast<size_t>(q0 + quad * 32);
#pragma unroll 1
                for (int seg = 0; seg < D / 64; ++seg) {
                    uint32_t r[2][32];
                    if (!empty) {
                        ptx::tmem_ld32(t_o + 64 * seg, r[0]);
                        ptx::tmem_ld32(t_o + 64 * seg + 32, r[1]);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int e = 0; e < 32; ++e) r[h][e] = 0u;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t *x = &r[u >> 2][8 * (u & 3)];
                        uint4 val;
                        val.x = ptx::pack_bf16x2(__uint_as_float(x[0]) * inv_l, __uint_as_float(x[1]) * inv_l);
                        val.y = ptx::pack_bf16x2(__uint_as_float(x[2]) * inv_l, __uint_as_float(x[3]) * inv_l);
                        val.z = ptx::pack_bf16x2(__uint_as_float(x[4]) * inv_l, __uint_as_float(x[5]) * inv_l);
                        val.w = ptx::pack_bf16x2(__uint_as_float(x[6]) * inv_l, __uint_as_float(x[7]) * inv_l);
                        ptx::st_shared_v4(stg + static_cast<uint32_t>(lane) * 128u +
                                              ((static_cast<uint32_t>(u) ^ sw) << 4),
                                          val);
                    }
                    __syncwarp();
#pragma unroll
                    for (int kq = 0; kq < 8; ++kq) {
                        const int wr = rr0 + 4 * kq;  // warp row
                        const uint4 val = ptx::ld_shared_v4(stg + static_cast<uint32_t>(wr) * 128u +
                                                            ((static_cast<uint32_t>(part) ^ static_cast<uint32_t>(wr & 7)) << 4));
                        const size_t gidx = rbase + static_cast<size_t>(wr);
                        if (q0 + quad * 32 + wr < p.N && ATTN_CHECK(gidx < rows_out, 7u))
                            reinterpret_cast<uint4 *>(p.o + gidx * D + seg * 64)[part] = val;
                    }
                    __syncwarp();
                }
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + ridx * D);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    if (!empty) {
                        ptx::tmem_ld32(t_o + 32 * c, r);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = 0u;
                    }
                    if (store_row) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            uint4 val;
                            val.x = ptx::pack_bf16x2(__uint_as_float(r[8 * g + 0]) * inv_l,
                                                     __uint_as_float(r[8 * g + 1]) * inv_l);
                            val.y = ptx::pack_bf16x2(__uint_as_float(r[8 * g + 2]) * inv_l,
                                                     __uint_as_float(r[8 * g + 3]) * inv_l);
                            val.z = ptx::pack_bf16x2(__uint_as_float(r[8 * g + 4]) * inv_l,
                                                     __uint_as_float(r[8 * g + 5]) * inv_l);
                            val.w = ptx::pack_bf16x2(__uint_as_float(r[8 * g + 6]) * inv_l,
                                                     __uint_as_float(r[8 * g + 7]) * inv_l);
                            dst[4 * c + g] = val;
                        }
                    }
                }
            }
            if (!ok) break;
            if (store_row) p.lse[ridx] = lse_nat;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Block quantisation to e4m3 (the FlashAttention-3 review's "Block Quantization": each
// B_r x d block gets its own scale from its largest magnitude, then the scaled values
// are rounded to FP8). One CTA per (block of 128 rows, head): amax = max |x|,
// inv = 448 / amax, code = e4m3(x * inv) rounded to nearest even with saturation, and
// scale = amax / 448; an all-zero block gets scale 1. The division and product are
// plain IEEE fp32 operations, so the codes are reproducible bit for bit.
template <int D>
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const __nv_bfloat16 *__restrict__ x,
                                                            uint8_t *__restrict__ codes,
                                                            float *__restrict__ scales, int N, int nblk) {
    constexpr int GROUPS = BM * D / 8 / 256;  // 8-element groups per thread
    const int blk = blockIdx.x, h = blockIdx.y;
    const int r0 = blk * BM;
    if (!ATTN_CHECK(r0 < N && blk < nblk, 40u)) return;
    const int n = min(BM, N - r0) * D;  // elements in this block
    const size_t base = (static_cast<size_t>(h) * N + r0) * D;
    uint4 v[GROUPS];
    float amax = 0.f;
#pragma unroll
    for (int g = 0; g < GROUPS; ++g) {
        const int e0 = (threadIdx.x + g * 256) * 8;
        if (e0 < n) {
            v[g] = *reinterpret_cast<const uint4 *>(x + base + e0);
            const uint32_t w[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
            }
        }
    }
    __shared__ float red[8];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    if (threadIdx.x == 0) scales[static_cast<size_t>(h) * nblk + blk] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
    for (int g = 0; g < GROUPS; ++g) {
        const int e0 = (threadIdx.x + g * 256) * 8;
        if (e0 < n) {
            const uint32_t w[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
            uint2 out;
            out.x = ptx::pack_e4m3x4(__fmul_rn(__uint_as_float(w[0] << 16), inv),
                                     __fmul_rn(__uint_as_float(w[0] & 0xFFFF0000u), inv),
                                     __fmul_rn(__uint_as_float(w[1] << 16), inv),
                                     __fmul_rn(__uint_as_float(w[1] & 0xFFFF0000u), inv));
            out.y = ptx::pack_e4m3x4(__fmul_rn(__uint_as_float(w[2] << 16), inv),
                                     __fmul_rn(__uint_as_float(w[2] & 0xFFFF0000u), inv),
                                     __fmul_rn(__uint_as_float(w[3] << 16), inv),
                                     __fmul_rn(__uint_as_float(w[3] & 0xFFFF0000u), inv));
            *reinterpret_cast<uint2 *>(codes + base + e0) = out;
        }
    }
}

// Incoherent processing, then block quantisation (the FlashAttention-3 review's FP8 path):
// the rows are rotated by the random orthogonal M = diag(s) H / sqrt(128), s = +-1 per
// channel and H the Sylvester Hadamard matrix of order 128, and the rotated block is
// quantised as above. One CTA per (block of 128 rows, head); a warp takes 4 rows at a
// time, 8 lanes per row, lane l holding elements 16 (l mod 8) .. 16 (l mod 8) + 15 of
// row l / 8. y = (x o s) H is formed in fp32 by the seven butterfly stages of the fast
// Walsh-Hadamard transform (element-index bits 0-3 inside a lane, bits 4-6 across the
// row's 8 lanes by shuffles). Codes are e4m3(y * (448 / amax)) and the block's scale is
// (amax / 448) / sqrt(128), so that code x scale approximates x M; an all-zero block
// gets scale 1.
__global__ void __launch_bounds__(256, 2) quantize_hadamard_e4m3_kernel(const __nv_bfloat16 *__restrict__ x,
                                                                     uint8_t *__restrict__ codes,
                                                                     float *__restrict__ scales, int N, int nblk,
                                                                     unsigned long long neg_lo,
                                                                     unsigned long long neg_hi) {
    constexpr int D = 128, PASSES = BM / 8 / 4;  // 8 warps x 4 rows per pass
    const int blk = blockIdx.x, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = lane & 7;  // which 16 channels of the row
    // channels 16 part .. 16 part + 15 whose sign is flipped (bit c of the 128-bit mask)
    const uint32_t neg = static_cast<uint32_t>((part < 4 ? neg_lo : neg_hi) >> (16 * (part & 3))) & 0xFFFFu;
    // the flips as XOR masks on the sign bits of the packed bf16 pairs (an exact negation)
    uint32_t flip[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        flip[i] = (((neg >> (2 * i)) & 1u) << 15) | (((neg >> (2 * i + 1)) & 1u) << 31);
    float y[PASSES][16];
    float amax = 0.f;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
        const int row = blk * BM + (warp * PASSES + ps) * 4 + (lane >> 3);
        float v[16];
        if (row < N) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (static_cast<size_t>(h) * N + row) * D + 16 * part);
            const uint4 w0 = src[0], w1 = src[1];
            const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t ws = w[i] ^ flip[i];
                v[2 * i] = __uint_as_float(ws << 16);
                v[2 * i + 1] = __uint_as_float(ws & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
        // index bits 0-3 inside the lane: pairs (i, i + 2^b) for i with bit b clear
#pragma unroll
        for (int b = 0; b < 4; ++b) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i & (1 << b)) continue;
                const float lo = v[i], hi = v[i + (1 << b)];
                v[i] = lo + hi;
                v[i + (1 << b)] = lo - hi;
            }
        }
        // index bits 4-6 = lane bits 0-2: the lane with the bit clear keeps x_i + x_j,
        // its partner x_i - x_j, both as one fma with a factor of +-1 (the same single
        // rounding as the sum or difference)
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const float sg = ((lane >> k) & 1) ? -1.f : 1.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float pv = __shfl_xor_sync(0xffffffffu, v[i], 1 << k);
                v[i] = fmaf(v[i], sg, pv);
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            y[ps][i] = v[i];
            if (row < N) amax = fmaxf(amax, fabsf(v[i]));
        }
    }
    __shared__ float red[8];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    if (threadIdx.x == 0)
        scales[static_cast<size_t>(h) * nblk + blk] =
            amax > 0.f ? __fmul_rn(__fdiv_rn(amax, 448.f), 0.0883883476483184f) : 1.f;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
        const int row = blk * BM + (warp * PASSES + ps) * 4 + (lane >> 3);
        if (row < N) {
            uint4 out;
            out.x = ptx::pack_e4m3x4(__fmul_rn(y[ps][0], inv), __fmul_rn(y[ps][1], inv), __fmul_rn(y[ps][2], inv),
                                     __fmul_rn(y[ps][3], inv));
            out.y = ptx::pack_e4m3x4(__fmul_rn(y[ps][4], inv), __fmul_rn(y[ps][5], inv), __fmul_rn(y[ps][6], inv),
                                     __fmul_rn(y[ps][7], inv));
            out.z = ptx::pack_e4m3x4(__fmul_rn(y[ps][8], inv), __fmul_rn(y[ps][9], inv),
                                     __fmul_rn(y[ps][10], inv), __fmul_rn(y[ps][11], inv));
            out.w = ptx::pack_e4m3x4(__fmul_rn(y[ps][12], inv), __fmul_rn(y[ps][13], inv),
                                     __fmul_rn(y[ps][14], inv), __fmul_rn(y[ps][15], inv));
            *reinterpret_cast<uint4 *>(codes + (static_cast<size_t>(h) * N + row) * D + 16 * part) = out;
        }
    }
}

// Decode shape, split key sequence: merge the per-split results of each packed query
// row. With lse_s and o_s (o_s normalised within split s), lse = ln sum_s exp(lse_s)
// and o = sum_s exp(lse_s - lse) o_s: the log-sum-exp merge of partial softmaxes
// (splits with no visible key carry lse_s = -inf and weigh nothing). One warp per row,
// each lane owning D / 32 consecutive columns.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const float *__restrict__ o_part,
                                                             const float *__restrict__ lse_part,
                                                             __nv_bfloat16 *__restrict__ o,
                                                             float *__restrict__ lse, int rows,
                                                             int splits) {
    constexpr int PER = D / 32;
    // launched as a programmatic dependent of the split kernel: the blocks may be resident
    // before it ends; this waits until it has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row = blockIdx.x * 8 + static_cast<int>(threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    if (!ATTN_CHECK(row >= 0 && splits >= 1, 30u)) return;
    // the loads of different splits are independent: unrolled so that they overlap
    float m = -INFINITY;
#pragma unroll 4
    for (int s = lane; s < splits; s += 32) m = fmaxf(m, lse_part[static_cast<size_t>(s) * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float sum = 0.f;
    if (m != -INFINITY) {
        for (int s = lane; s < splits; s += 32) {
            const float l = lse_part[static_cast<size_t>(s) * rows + row];
            if (l != -INFINITY) sum += expf(l - m);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float lse_row = (m == -INFINITY) ? -INFINITY : m + logf(sum);
    float acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] = 0.f;
    if (m != -INFINITY) {
#pragma unroll 4
        for (int s = 0; s < splits; ++s) {
            const float l = lse_part[static_cast<size_t>(s) * rows + row];
            if (l == -INFINITY) continue;
            const float wgt = expf(l - lse_row);
            const float *src = o_part + (static_cast<size_t>(s) * rows + row) * D + lane * PER;
            if constexpr (PER == 4) {
                const float4 x = *reinterpret_cast<const float4 *>(src);
                acc[0] = fmaf(wgt, x.x, acc[0]);
                acc[1] = fmaf(wgt, x.y, acc[1]);
                acc[2] = fmaf(wgt, x.z, acc[2]);
                acc[3] = fmaf(wgt, x.w, acc[3]);
            } else {
                const float2 x = *reinterpret_cast<const float2 *>(src);
                acc[0] = fmaf(wgt, x.x, acc[0]);
                acc[1] = fmaf(wgt, x.y, acc[1]);
            }
        }
    }
    uint32_t *dst = reinterpret_cast<uint32_t *>(o + static_cast<size_t>(row) * D + lane * PER);
#pragma unroll
    for (int c = 0; c < PER / 2; ++c) dst[c] = ptx::pack_bf16x2(acc[2 * c], acc[2 * c + 1]);
    if (lane == 0) lse[row] = lse_row;
}

#ifdef ATTN_DEBUG
// One failed check at site 99 (nothing is accessed): exercises the debug build's
// reporting path.
__global__ void debug_selftest_kernel() {
    if (threadIdx.x == 0) (void)ATTN_CHECK(false, 99u);
}
#endif

// One warp waits on a barrier nothing will complete; exercises the timeout path.
__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    wait_warp(ptx::smem_addr(&bar), 0u, &abort_flag, limit_ns);
}

#include "attn_bwd.cuh"

}  // namespace attn

// ====================================================================== host side
namespace {

using attn::Cfg;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready;
    bool bwd_ready;
    int sms;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Streams and events of attn_fwd_host's copy pipeline, created once per device on the
// first call and kept until the process exits.
constexpr int HOST_CHUNKS = 8;
struct HostPipe {
    std::mutex mu;               // one enqueue sequence at a time
    cudaStream_t h2d, d2h;       // non-blocking: no implicit ordering with the legacy stream
    cudaEvent_t start, done, in[HOST_CHUNKS], out[HOST_CHUNKS];
};
HostPipe *g_host_pipe[kMaxDevices];
thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return ATTN_ERR_CUDA;
}

EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// per-device one-time set-up: architecture check, SM count, shared-memory opt-in
int device_setup(int *sms_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &di = g_dev[dev];
    if (!di.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
        // the warpgroup register split must fit in what a CTA is launched with;
        // otherwise setmaxnreg.inc would wait for registers that never come
        const void *kernels[5] = {reinterpret_cast<const void *>(attn::attn_fwd_kernel<64, false, false>),
                                  reinterpret_cast<const void *>(attn::attn_fwd_kernel<128, false, false>),
                                  reinterpret_cast<const void *>(attn::attn_fwd_kernel<64, true, false>),
                                  reinterpret_cast<const void *>(attn::attn_fwd_kernel<128, true, false>),
                                  reinterpret_cast<const void *>(attn::attn_fwd_kernel<128, false, true>)};
        for (const void *kfn : kernels) {
            cudaFuncAttributes fa;
            if ((e = cudaFuncGetAttributes(&fa, kfn)) != cudaSuccess) return cuda_fail(e);
            if (fa.numRegs * attn::NUM_THREADS <
                2 * 128 * attn::SOFTMAX_REGS + 128 * attn::PRODUCER_REGS)
                return ATTN_ERR_UNSUPPORTED;
        }
        if ((e = cudaFuncSetAttribute(attn::attn_fwd_kernel<64, false, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<64>::SMEM_ALLOC)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn::attn_fwd_kernel<128, false, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<128>::SMEM_ALLOC)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn::attn_fwd_kernel<64, true, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<64, false, true>::SMEM_ALLOC)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn::attn_fwd_kernel<128, true, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<128, false, true>::SMEM_ALLOC)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn::attn_fwd_kernel<128, false, true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<128, true>::SMEM_ALLOC)) != cudaSuccess)
            return cuda_fail(e);
        di.sms = sms;
        di.ready = true;
    }
    *sms_out = di.sms;
    return ATTN_OK;
}

bool misaligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) != 0; }

int validate(const void *q, const void *k, const void *v, const void *o, const float *lse, int B,
             int Hq, int Hkv, int N, int d, int causal, int window, float scale) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULLPTR;
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || window < 0) return ATTN_ERR_SHAPE;
    if (Hq % Hkv != 0) return ATTN_ERR_SHAPE;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_SHAPE;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (causal != 0 && causal != 1) return ATTN_ERR_SHAPE;
    // index range: rows fit 32-bit tile arithmetic; unit count fits int
    if (N > (1 << 30)) return ATTN_ERR_SHAPE;
    const long long bh = static_cast<long long>(B) * Hq;
    const long long n_pairs = ((N + attn::BM - 1) / attn::BM + 1) / 2;
    if (bh > INT_MAX || bh * n_pairs > INT_MAX) return ATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * Hkv > INT_MAX) return ATTN_ERR_SHAPE;
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
        misaligned(lse, 4))
        return ATTN_ERR_ALIGN;
    return ATTN_OK;
}

int encode_map_u8(EncodeTiledFn enc, CUtensorMap *map, const void *base, int d, int N, long long BH) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d),
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d)};
    cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(attn::BM), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return ATTN_OK;
}

// bf16 [BH, N, d] as boxes of `rows` rows x 64 columns (128 bytes), 128-byte swizzled
int encode_map(EncodeTiledFn enc, CUtensorMap *map, const void *base, int d, int N, long long BH,
               int rows = attn::BM) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2u,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2u};
    cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return ATTN_OK;
}

template <int D>
int launch(const void *q, const void *k, const void *v, void *o, float *o32, float *lse, const int *key_len,
           int B, int Hq, int Hkv, int N, int causal, int window, float scale, cudaStream_t stream,
           int sms) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return cuda_fail(cudaErrorNotSupported);
    CUtensorMap mq, mk, mv;
    int rc;
    if ((rc = encode_map(enc, &mq, q, D, N, static_cast<long long>(B) * Hq)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mk, k, D, N, static_cast<long long>(B) * Hkv)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mv, v, D, N, static_cast<long long>(B) * Hkv)) != ATTN_OK) return rc;
    attn::Params p;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.key_len = key_len;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.N = N;
    p.group = Hq / Hkv;
    p.causal = causal;
    // a window of N or more keys excludes nothing: run it as no window (same result)
    p.window = window >= N ? 0 : window;
    p.sym = (p.window > 0 && !causal) ? 1 : 0;
    p.n_kv = (N + attn::BN - 1) / attn::BN;
    p.n_pairs = (p.n_kv + 1) / 2;
    p.num_units = B * Hq * p.n_pairs;
    p.sl2 = scale * 1.4426950408889634f;
    p.timeout_ns = attn::WAIT_LIMIT_NS;
    p.div_bh = attn::make_fastdiv(static_cast<uint32_t>(B * Hq));
    p.div_hq = attn::make_fastdiv(static_cast<uint32_t>(Hq));
    p.div_group = attn::make_fastdiv(static_cast<uint32_t>(p.group));
    p.Nk = N;
    p.pos_off = 0;
    p.Nq = N;
    p.splits = 1;
    p.split_lo = p.split_len = p.split_hi = 0;
    p.div_splits = attn::make_fastdiv(1u);
    p.div_nq = attn::make_fastdiv(1u);
    p.dec2 = 0;
    p.o_part = p.lse_part = nullptr;
    p.o32 = o32;
    p.q_scale = p.k_scale = p.v_scale = nullptr;
    const int grid = p.num_units < sms ? p.num_units : sms;
    cudaError_t e = attn::launch_fwd_kernel<D, false, false>(grid, Cfg<D>::SMEM_ALLOC, stream, mq, mk, mv, p);
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

// e4m3 operands with block scales (d = 128, plain forward)
int launch_fp8(const void *q8, const void *k8, const void *v8, const float *qs, const float *ks,
               const float *vs, void *o, float *lse, int B, int Hq, int Hkv, int N, int causal, int window,
               float scale, cudaStream_t stream, int sms) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return cuda_fail(cudaErrorNotSupported);
    CUtensorMap mq, mk, mv;
    int rc;
    if ((rc = encode_map_u8(enc, &mq, q8, 128, N, static_cast<long long>(B) * Hq)) != ATTN_OK) return rc;
    if ((rc = encode_map_u8(enc, &mk, k8, 128, N, static_cast<long long>(B) * Hkv)) != ATTN_OK) return rc;
    if ((rc = encode_map_u8(enc, &mv, v8, 128, N, static_cast<long long>(B) * Hkv)) != ATTN_OK) return rc;
    attn::Params p;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.key_len = nullptr;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.N = N;
    p.group = Hq / Hkv;
    p.causal = causal;
    p.window = window >= N ? 0 : window;
    p.sym = (p.window > 0 && !causal) ? 1 : 0;
    p.n_kv = (N + attn::BN - 1) / attn::BN;
    p.n_pairs = (p.n_kv + 1) / 2;
    p.num_units = B * Hq * p.n_pairs;
    p.sl2 = scale * 1.4426950408889634f;
    p.timeout_ns = attn::WAIT_LIMIT_NS;
    p.div_bh = attn::make_fastdiv(static_cast<uint32_t>(B * Hq));
    p.div_hq = attn::make_fastdiv(static_cast<uint32_t>(Hq));
    p.div_group = attn::make_fastdiv(static_cast<uint32_t>(p.group));
    p.Nk = N;
    p.pos_off = 0;
    p.Nq = N;
    p.splits = 1;
    p.split_lo = p.split_len = p.split_hi = 0;
    p.div_splits = attn::make_fastdiv(1u);
    p.div_nq = attn::make_fastdiv(1u);
    p.dec2 = 0;
    p.o_part = p.lse_part = nullptr;
    p.o32 = nullptr;
    p.q_scale = qs;
    p.k_scale = ks;
    p.v_scale = vs;
    const int grid = p.num_units < sms ? p.num_units : sms;
    cudaError_t e = attn::launch_fwd_kernel<128, false, true>(grid, Cfg<128, true>::SMEM_ALLOC, stream, mq, mk, mv, p);
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

// Split count for the decode shape: units are (batch * Hkv, split) pairs run one per CTA
// at a time on `sms` CTAs; the makespan is about rounds x (key tiles per split + the
// per-unit cost of loading Q, filling the pipeline and writing the partial result,
// about two tiles' worth). Take the count that minimises it.
int choose_splits(long long bhkv, int kv_tiles, int sms) {
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= kv_tiles && s <= 256; ++s) {
        const long long rounds = (bhkv * s + sms - 1) / sms;
        const long long per_unit = (kv_tiles + s - 1) / s + 2;
        const long long cost = rounds * per_unit;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Device address of the static scratch array on the current device. The first call on
// a device looks it up (cudaGetSymbolAddress, with that device current) and caches it.
int noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if ((e = cudaGetSymbolAddress(&ptr, attn::g_noalloc_scratch)) != cudaSuccess) return cuda_fail(e);
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}

// attn_fwd_host's streams and events on the current device, created on first use
int host_pipe(HostPipe **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_host_pipe[dev]) {
        HostPipe *hp = new HostPipe();
        const unsigned ev_flags = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&hp->h2d, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp->start, ev_flags)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp->done, ev_flags)) != cudaSuccess)
            return cuda_fail(e);
        for (int c = 0; c < HOST_CHUNKS; ++c)
            if ((e = cudaEventCreateWithFlags(&hp->in[c], ev_flags)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp->out[c], ev_flags)) != cudaSuccess)
                return cuda_fail(e);
        g_host_pipe[dev] = hp;
    }
    *out = g_host_pipe[dev];
    return ATTN_OK;
}

size_t decode_workspace(long long rows, int d, int splits) {
    if (splits <= 1) return 0;
    const size_t o_bytes = static_cast<size_t>(splits) * static_cast<size_t>(rows) * d * sizeof(float);
    const size_t o_pad = (o_bytes + 255) / 256 * 256;
    return o_pad + static_cast<size_t>(splits) * static_cast<size_t>(rows) * sizeof(float);
}

int validate_decode(const void *q, const void *k, const void *v, const void *o, const float *lse, int B,
                    int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window, float scale) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULLPTR;
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < Nq || window < 0) return ATTN_ERR_SHAPE;
    if (Hq % Hkv != 0) return ATTN_ERR_SHAPE;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_SHAPE;
    if (causal != 0 && causal != 1) return ATTN_ERR_SHAPE;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(Hq / Hkv) * Nq > attn::BM) return ATTN_ERR_UNSUPPORTED;  // one packed tile
    if (Nk > (1 << 30)) return ATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * Hkv * 256 > INT_MAX) return ATTN_ERR_SHAPE;
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
        misaligned(lse, 4))
        return ATTN_ERR_ALIGN;
    return ATTN_OK;
}

template <int D>
int launch_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int causal, int window, float scale, int splits,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream, int sms) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return cuda_fail(cudaErrorNotSupported);
    const int G = Hq / Hkv;
    const int R = G * Nq;  // packed query rows per KV head
    const long long bhkv = static_cast<long long>(B) * Hkv;
    const int kv_tiles = (Nk + attn::BN - 1) / attn::BN;
    if (splits <= 0) splits = choose_splits(bhkv, kv_tiles, sms);
    if (splits > kv_tiles) splits = kv_tiles;
    const long long rows = bhkv * R;
    if (splits > 1) {
        if (!workspace) return ATTN_ERR_NULLPTR;
        if (misaligned(workspace, 256)) return ATTN_ERR_ALIGN;
        if (workspace_bytes < decode_workspace(rows, D, splits)) return ATTN_ERR_WORKSPACE;
    }
    CUtensorMap mq, mk, mv;
    int rc;
    if ((rc = encode_map(enc, &mq, q, D, R, bhkv)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mk, k, D, Nk, bhkv)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mv, v, D, Nk, bhkv)) != ATTN_OK) return rc;
    attn::Params p;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.key_len = nullptr;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.N = R;
    p.group = G;
    p.causal = causal;
    p.window = window >= Nk ? 0 : window;
    p.sym = (p.window > 0 && !causal) ? 1 : 0;
    p.n_kv = kv_tiles;
    p.n_pairs = 1;
    p.sl2 = scale * 1.4426950408889634f;
    p.timeout_ns = attn::WAIT_LIMIT_NS;
    p.div_bh = p.div_hq = p.div_group = attn::make_fastdiv(1u);
    p.Nk = Nk;
    p.pos_off = Nk - Nq;
    p.Nq = Nq;
    p.splits = splits;
    // key tiles some packed row can see: from the earliest query's window start to the end
    const int pos_min = Nk - Nq;
    const int first_key = p.window > 0 ? (pos_min - p.window + 1 > 0 ? pos_min - p.window + 1 : 0) : 0;
    p.split_lo = first_key / attn::BN;
    p.split_hi = kv_tiles;
    p.split_len = (p.split_hi - p.split_lo + splits - 1) / splits;
    p.div_splits = attn::make_fastdiv(static_cast<uint32_t>(splits));
    p.div_nq = attn::make_fastdiv(static_cast<uint32_t>(Nq));
    // both query tiles on each split when the packed rows fit one warp's 32 lanes and the
    // split is long enough (8 key tiles or more per tile) to pay for the exchange between
    // the tiles at its end
    p.dec2 = (R <= 32 && p.split_len >= 16) ? 1 : 0;
    p.num_units = static_cast<int>(bhkv * splits);
    p.q_scale = p.k_scale = p.v_scale = nullptr;
    p.o32 = nullptr;
    if (splits > 1) {
        p.o_part = static_cast<float *>(workspace);
        const size_t o_bytes = static_cast<size_t>(splits) * static_cast<size_t>(rows) * D * sizeof(float);
        p.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + (o_bytes + 255) / 256 * 256);
    } else {
        p.o_part = p.lse_part = nullptr;
    }
    const int grid = p.num_units < sms ? p.num_units : sms;
    cudaError_t e = attn::launch_fwd_kernel<D, true, false>(grid, Cfg<D, false, true>::SMEM_ALLOC, stream, mq, mk, mv, p);
    if (e != cudaSuccess) return cuda_fail(e);
    if (splits > 1) {
        // a programmatic dependent launch: its blocks can take SMs as split CTAs finish,
        // instead of waiting for the whole grid to drain before being launched
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
        lc.blockDim = dim3(256);
        lc.dynamicSmemBytes = 0;
        lc.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute la[1];
        la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        la[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = la;
        lc.numAttrs = 1;
        e = cudaLaunchKernelEx(&lc, attn::decode_combine_kernel<D>, static_cast<const float *>(p.o_part),
                               static_cast<const float *>(p.lse_part), static_cast<__nv_bfloat16 *>(o), lse,
                               static_cast<int>(rows), splits);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return ATTN_OK;
}


// ------------------------------------------------------------------ backward
// one-time shared-memory opt-in of the backward kernels on the current device
int bwd_setup(int *sms_out) {
    int rc = device_setup(sms_out);
    if (rc != ATTN_OK) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &di = g_dev[dev];
    if (!di.bwd_ready) {
        if ((e = cudaFuncSetAttribute(attn::attn_bwd_kernel<64, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      attn::BwdCfg<64>::SMEM_ALLOC)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn::attn_bwd_kernel<64, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      attn::BwdCfg<64>::SMEM_ALLOC)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn::attn_bwd_kernel<128, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      attn::BwdCfg<128>::SMEM_ALLOC)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn::attn_bwd_kernel<128, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      attn::BwdCfg<128>::SMEM_ALLOC)) != cudaSuccess)
            return cuda_fail(e);
        di.bwd_ready = true;
    }
    return ATTN_OK;
}

// workspace of the backward: lse log2(e), then D = rowsum(dO o O), of every query row
// (fp32), each head's rows padded to a multiple of the tile
long long bwd_n_pad(int N) { return (static_cast<long long>(N) + attn::BM - 1) / attn::BM * attn::BM; }
size_t bwd_workspace(int B, int Hq, int N) {
    return 2 * static_cast<size_t>(B) * Hq * bwd_n_pad(N) * sizeof(float);
}

template <int D>
int launch_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
               const void *dout, void *dq, void *dk, void *dv, const int *key_len, int B, int Hq, int Hkv,
               int N, int causal, int window, float scale, void *workspace, cudaStream_t stream, int sms) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return cuda_fail(cudaErrorNotSupported);
    const long long BHq = static_cast<long long>(B) * Hq, BHkv = static_cast<long long>(B) * Hkv;
    // 128-row boxes for the stationary operands, 64-row boxes for the streamed ones
    CUtensorMap mq, mk, mv, mdo, mq64, mk64, mv64, mdo64;
    int rc;
    if ((rc = encode_map(enc, &mq, q, D, N, BHq)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mk, k, D, N, BHkv)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mv, v, D, N, BHkv)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mdo, dout, D, N, BHq)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mq64, q, D, N, BHq, 64)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mk64, k, D, N, BHkv, 64)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mv64, v, D, N, BHkv, 64)) != ATTN_OK) return rc;
    if ((rc = encode_map(enc, &mdo64, dout, D, N, BHq, 64)) != ATTN_OK) return rc;
    const int n_pad = static_cast<int>(bwd_n_pad(N));
    float *lse2 = static_cast<float *>(workspace);
    float *dsum = lse2 + BHq * n_pad;
    // lse log2(e) and D = rowsum(dO o O): warps of pre_rows_per_warp<D>() padded rows, 8 per block
    const long long prows = BHq * n_pad;
    const long long pre_warps = prows / attn::pre_rows_per_warp<D>();
    attn::bwd_preprocess_kernel<D><<<static_cast<unsigned>((pre_warps + 7) / 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse, lse2, dsum, BHq, N,
        n_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    attn::BwdParams p;
    p.lse2 = lse2;
    p.dsum = dsum;
    p.dq = static_cast<__nv_bfloat16 *>(dq);
    p.dk = static_cast<__nv_bfloat16 *>(dk);
    p.dv = static_cast<__nv_bfloat16 *>(dv);
    p.key_len = key_len;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.N = N;
    p.N_pad = n_pad;
    p.group = Hq / Hkv;
    p.causal = causal;
    p.window = window >= N ? 0 : window;  // a window of N or more keys excludes nothing
    p.sym = (p.window > 0 && !causal) ? 1 : 0;
    p.n_kv = (N + attn::BN - 1) / attn::BN;
    p.sl2 = scale * 1.4426950408889634f;
    p.scale = scale;
    p.timeout_ns = attn::WAIT_LIMIT_NS;
    p.div_bhkv = attn::make_fastdiv(static_cast<uint32_t>(BHkv));
    p.div_hkv = attn::make_fastdiv(static_cast<uint32_t>(Hkv));
    p.div_bhq = attn::make_fastdiv(static_cast<uint32_t>(BHq));
    p.div_hq = attn::make_fastdiv(static_cast<uint32_t>(Hq));
    p.div_group = attn::make_fastdiv(static_cast<uint32_t>(p.group));
    // dK, dV: one unit per (key tile, batch, kv head)
    p.num_units = static_cast<int>(BHkv * p.n_kv);
    int grid = p.num_units < sms ? p.num_units : sms;
    // both kernels are programmatic dependents of the kernel before them (see the kernel's
    // prologue): each starts its prologue while the previous one finishes
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc = {};
    lc.blockDim = dim3(attn::BWD_THREADS);
    lc.dynamicSmemBytes = attn::BwdCfg<D>::SMEM_ALLOC;
    lc.stream = static_cast<cudaStream_t>(stream);
    lc.attrs = la;
    lc.numAttrs = 1;
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    e = cudaLaunchKernelEx(&lc, attn::attn_bwd_kernel<D, 0>, mk, mv, mq64, mdo64, p);
    if (e != cudaSuccess) return cuda_fail(e);
    // dQ: one unit per (query tile, batch, query head)
    p.num_units = static_cast<int>(BHq * p.n_kv);
    grid = p.num_units < sms ? p.num_units : sms;
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    e = cudaLaunchKernelEx(&lc, attn::attn_bwd_kernel<D, 1>, mq, mdo, mk64, mv64, p);
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

}  // namespace

extern "C" {

// o: bf16 output, or (o32 set) the fp32 output; exactly one of the two is written
static int fwd_common(const void *q, const void *k, const void *v, void *o, float *o32, float *lse,
                      const int *key_len, int B, int Hq, int Hkv, int N, int d, int causal,
                      int window, float scale, void *stream) {
    int rc = validate(q, k, v, o32 ? static_cast<const void *>(o32) : o, lse, B, Hq, Hkv, N, d, causal,
                      window, scale);
    if (rc != ATTN_OK) return rc;
    int sms = 0;
    if ((rc = device_setup(&sms)) != ATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d == 64) return launch<64>(q, k, v, o, o32, lse, key_len, B, Hq, Hkv, N, causal, window, scale, s, sms);
    return launch<128>(q, k, v, o, o32, lse, key_len, B, Hq, Hkv, N, causal, window, scale, s, sms);
}

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv,
             int N, int d, int causal, int window, float scale, void *stream) {
    return fwd_common(q, k, v, o, nullptr, lse, nullptr, B, Hq, Hkv, N, d, causal, window, scale, stream);
}

int attn_fwd_o32(const void *q, const void *k, const void *v, float *o32, float *lse, const int *key_len,
                 int B, int Hq, int Hkv, int N, int d, int causal, int window, float scale, void *stream) {
    if (!o32) return ATTN_ERR_NULLPTR;
    if (key_len && misaligned(key_len, 4)) return ATTN_ERR_ALIGN;
    return fwd_common(q, k, v, nullptr, o32, lse, key_len, B, Hq, Hkv, N, d, causal, window, scale, stream);
}

int attn_fwd_padded(const void *q, const void *k, const void *v, void *o, float *lse,
                    const int *key_len, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                    float scale, void *stream) {
    if (!key_len) return ATTN_ERR_NULLPTR;
    if (misaligned(key_len, 4)) return ATTN_ERR_ALIGN;
    return fwd_common(q, k, v, o, nullptr, lse, key_len, B, Hq, Hkv, N, d, causal, window, scale, stream);
}

size_t attn_fwd_decode_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int splits) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < Nq || Hq % Hkv != 0 || (d != 64 && d != 128))
        return 0;
    const int kv_tiles = (Nk + attn::BN - 1) / attn::BN;
    const long long bhkv = static_cast<long long>(B) * Hkv;
    if (splits <= 0) {
        int sms = 0;
        if (device_setup(&sms) != ATTN_OK) return 0;
        splits = choose_splits(bhkv, kv_tiles, sms);
    }
    if (splits > kv_tiles) splits = kv_tiles;
    return decode_workspace(bhkv * (Hq / Hkv) * Nq, d, splits);
}

int attn_fwd_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                    int Hkv, int Nq, int Nk, int d, int causal, int window, float scale, int splits,
                    void *workspace, size_t workspace_bytes, void *stream) {
    int rc = validate_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, window, scale);
    if (rc != ATTN_OK) return rc;
    int sms = 0;
    if ((rc = device_setup(&sms)) != ATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d == 64)
        return launch_decode<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, causal, window, scale, splits,
                                 workspace, workspace_bytes, s, sms);
    return launch_decode<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, causal, window, scale, splits,
                              workspace, workspace_bytes, s, sms);
}

int attn_fwd_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                            int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window, float scale,
                            int splits, void *stream) {
    int rc = validate_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, window, scale);
    if (rc != ATTN_OK) return rc;
    int sms = 0;
    if ((rc = device_setup(&sms)) != ATTN_OK) return rc;
    void *scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != ATTN_OK) return rc;
    // the same split count attn_fwd_decode would use; its partial results must fit
    const int kv_tiles = (Nk + attn::BN - 1) / attn::BN;
    const long long bhkv = static_cast<long long>(B) * Hkv;
    if (splits <= 0) splits = choose_splits(bhkv, kv_tiles, sms);
    if (splits > kv_tiles) splits = kv_tiles;
    if (decode_workspace(bhkv * (Hq / Hkv) * Nq, d, splits) > attn::NOALLOC_SCRATCH_BYTES)
        return ATTN_ERR_SCRATCH_LIMIT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d == 64)
        return launch_decode<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, causal, window, scale, splits,
                                 scratch, attn::NOALLOC_SCRATCH_BYTES, s, sms);
    return launch_decode<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, causal, window, scale, splits,
                              scratch, attn::NOALLOC_SCRATCH_BYTES, s, sms);
}

int attn_quantize_e4m3(const void *x, void *codes, float *scales, int BH, int N, int d, void *stream) {
    if (!x || !codes || !scales) return ATTN_ERR_NULLPTR;
    if (BH < 1 || N < 1 || N > (1 << 30)) return ATTN_ERR_SHAPE;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (misaligned(x, 16) || misaligned(codes, 8) || misaligned(scales, 4)) return ATTN_ERR_ALIGN;
    const int nblk = (N + attn::BM - 1) / attn::BM;
    if (static_cast<long long>(BH) > 65535) return ATTN_ERR_SHAPE;  // grid y
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>(nblk), static_cast<unsigned>(BH));
    if (d == 128)
        attn::quantize_e4m3_kernel<128><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(x),
                                                              static_cast<uint8_t *>(codes), scales, N, nblk);
    else
        attn::quantize_e4m3_kernel<64><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(x),
                                                             static_cast<uint8_t *>(codes), scales, N, nblk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

int attn_quantize_e4m3_hadamard(const void *x, uint64_t neg_lo, uint64_t neg_hi, void *codes, float *scales,
                                int BH, int N, int d, void *stream) {
    if (!x || !codes || !scales) return ATTN_ERR_NULLPTR;
    if (BH < 1 || N < 1 || N > (1 << 30)) return ATTN_ERR_SHAPE;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    if (misaligned(x, 16) || misaligned(codes, 16) || misaligned(scales, 4)) return ATTN_ERR_ALIGN;
    const int nblk = (N + attn::BM - 1) / attn::BM;
    if (static_cast<long long>(BH) > 65535) return ATTN_ERR_SHAPE;  // grid y
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>(nblk), static_cast<unsigned>(BH));
    attn::quantize_hadamard_e4m3_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(x),
                                                             static_cast<uint8_t *>(codes), scales, N, nblk,
                                                             static_cast<unsigned long long>(neg_lo),
                                                             static_cast<unsigned long long>(neg_hi));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

int attn_fwd_fp8(const void *q8, const void *k8, const void *v8, const float *q_scale, const float *k_scale,
                 const float *v_scale, void *o, float *lse, int B, int Hq, int Hkv, int N, int d, int causal,
                 int window, float scale, void *stream) {
    if (!q_scale || !k_scale || !v_scale) return ATTN_ERR_NULLPTR;
    int rc = validate(q8, k8, v8, o, lse, B, Hq, Hkv, N, d, causal, window, scale);
    if (rc != ATTN_OK) return rc;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    if (misaligned(q_scale, 4) || misaligned(k_scale, 4) || misaligned(v_scale, 4)) return ATTN_ERR_ALIGN;
    int sms = 0;
    if ((rc = device_setup(&sms)) != ATTN_OK) return rc;
    return launch_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, Hq, Hkv, N, causal, window, scale,
                      static_cast<cudaStream_t>(stream), sms);
}

int attn_fwd_host(const void *hq, const void *hk, const void *hv, void *ho, float *hlse, void *dq,
                  void *dk, void *dv, void *do_, float *dlse, int B, int Hq, int Hkv, int N, int d,
                  int causal, int window, float scale, void *stream) {
    int rc = validate(dq, dk, dv, do_, dlse, B, Hq, Hkv, N, d, causal, window, scale);
    if (rc != ATTN_OK) return rc;
    rc = validate(hq, hk, hv, ho, hlse, B, Hq, Hkv, N, d, causal, window, scale);
    if (rc != ATTN_OK) return rc;
    int sms = 0;
    if ((rc = device_setup(&sms)) != ATTN_OK) return rc;
    HostPipe *hp = nullptr;
    if ((rc = host_pipe(&hp)) != ATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The (batch, KV head) groups are independent, and each is contiguous in every
    // tensor: G query heads of q, o and lse, one head of k and v. Chunks of consecutive
    // groups go through a three-stage pipeline: host-to-device copies on one
    // library stream, the kernel on `stream`, device-to-host copies on a second library
    // stream, so that the copies of one chunk overlap the kernel and the copies of
    // the others. Each chunk is an attn_fwd call over its groups (one KV head each).
    const int G = Hq / Hkv;
    const long long groups = static_cast<long long>(B) * Hkv;
    const int nchunks = static_cast<int>(groups < HOST_CHUNKS ? groups : HOST_CHUNKS);
    const size_t q_g = static_cast<size_t>(G) * N * d * 2, kv_g = static_cast<size_t>(N) * d * 2;
    const size_t lse_g = static_cast<size_t>(G) * N * sizeof(float);
    auto at = [](const void *base, size_t off) { return static_cast<const char *>(base) + off; };
    auto atw = [](void *base, size_t off) { return static_cast<char *>(base) + off; };
    // one enqueue sequence at a time on the shared library streams and events
    std::lock_guard<std::mutex> lock(hp->mu);
    cudaError_t e;
    if ((e = cudaEventRecord(hp->start, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->h2d, hp->start, 0)) != cudaSuccess)
        return cuda_fail(e);
    for (int c = 0; c < nchunks; ++c) {
        const long long g0 = groups * c / nchunks, g1 = groups * (c + 1) / nchunks;
        const size_t ng = static_cast<size_t>(g1 - g0);
        const size_t oq = static_cast<size_t>(g0) * q_g, okv = static_cast<size_t>(g0) * kv_g;
        const size_t ol = static_cast<size_t>(g0) * lse_g;
        if ((e = cudaMemcpyAsync(atw(dq, oq), at(hq, oq), ng * q_g, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(dk, okv), at(hk, okv), ng * kv_g, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(dv, okv), at(hv, okv), ng * kv_g, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess ||
            (e = cudaEventRecord(hp->in[c], hp->h2d)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(s, hp->in[c], 0)) != cudaSuccess)
            return cuda_fail(e);
        rc = attn_fwd(atw(dq, oq), atw(dk, okv), atw(dv, okv), atw(do_, oq),
                      reinterpret_cast<float *>(atw(dlse, ol)), static_cast<int>(ng), G, 1, N, d, causal, window,
                      scale, stream);
        if (rc != ATTN_OK) return rc;
        if ((e = cudaEventRecord(hp->out[c], s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hp->d2h, hp->out[c], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(ho, oq), at(do_, oq), ng * q_g, cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(hlse, ol), at(dlse, ol), ng * lse_g, cudaMemcpyDeviceToHost, hp->d2h)) !=
                cudaSuccess)
            return cuda_fail(e);
    }
    // `stream` completes only after the last device-to-host copy
    if ((e = cudaEventRecord(hp->done, hp->d2h)) != cudaSuccess || (e = cudaStreamWaitEvent(s, hp->done, 0)) != cudaSuccess)
        return cuda_fail(e);
    return ATTN_OK;
}

size_t attn_bwd_workspace_size(int B, int Hq, int N, int d) {
    if (B < 1 || Hq < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    return bwd_workspace(B, Hq, N);
}

int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
             void *dq, void *dk, void *dv, const int *key_len, int B, int Hq, int Hkv, int N, int d, int causal,
             int window, float scale, void *workspace, size_t workspace_bytes, void *stream) {
    if (!dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_NULLPTR;
    int rc = validate(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window, scale);
    if (rc != ATTN_OK) return rc;
    const long long units = static_cast<long long>(B) * Hq * ((N + attn::BN - 1) / attn::BN);
    if (units > INT_MAX || static_cast<long long>(B) * Hq * bwd_n_pad(N) > INT_MAX) return ATTN_ERR_SHAPE;
    if (misaligned(dout, 16) || misaligned(dq, 16) || misaligned(dk, 16) || misaligned(dv, 16) ||
        misaligned(workspace, 256) || (key_len && misaligned(key_len, 4)))
        return ATTN_ERR_ALIGN;
    if (workspace_bytes < bwd_workspace(B, Hq, N)) return ATTN_ERR_WORKSPACE;
    int sms = 0;
    if ((rc = bwd_setup(&sms)) != ATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d == 64)
        return launch_bwd<64>(q, k, v, o, lse, dout, dq, dk, dv, key_len, B, Hq, Hkv, N, causal, window, scale,
                              workspace, s, sms);
    return launch_bwd<128>(q, k, v, o, lse, dout, dq, dk, dv, key_len, B, Hq, Hkv, N, causal, window, scale,
                           workspace, s, sms);
}

const char *attn_status_str(int status) {
    switch (status) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_NULLPTR: return "ATTN_ERR_NULLPTR: a required pointer is NULL";
        case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN: a buffer is not suitably aligned";
        case ATTN_ERR_SHAPE: return "ATTN_ERR_SHAPE: invalid sizes, window or scale";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: head dim, mask or device not supported";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: a CUDA runtime call failed";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a kernel wait ran out of time";
        case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: the workspace is smaller than required";
        case ATTN_ERR_SCRATCH_LIMIT:
            return "ATTN_ERR_SCRATCH_LIMIT: the split results need more than the fixed 8 MiB scratch";
        case ATTN_ERR_BOUNDS: return "ATTN_ERR_BOUNDS: an index check of the debug build failed";
        default: return "unknown attn_status";
    }
}

int attn_last_cuda_error(void) { return t_last_cuda_error; }

int attn_device_error(int clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int word = 0;
    if ((e = cudaMemcpyFromSymbol(&word, attn::g_status, sizeof word)) != cudaSuccess) return cuda_fail(e);
    if (clear) {
        const unsigned int zero = 0;
        if ((e = cudaMemcpyToSymbol(attn::g_status, &zero, sizeof zero)) != cudaSuccess) return cuda_fail(e);
    }
    if (word & attn::STATUS_BOUNDS) return ATTN_ERR_BOUNDS;
    return (word & attn::STATUS_TIMEOUT) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

int attn_debug_build(void) {
#ifdef ATTN_DEBUG
    return 1;
#else
    return 0;
#endif
}

int attn_debug_first_site(int clear) {
#ifdef ATTN_DEBUG
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int site = 0;
    if ((e = cudaMemcpyFromSymbol(&site, attn::g_debug_site, sizeof site)) != cudaSuccess) return cuda_fail(e);
    if (clear) {
        const unsigned int zero = 0;
        if ((e = cudaMemcpyToSymbol(attn::g_debug_site, &zero, sizeof zero)) != cudaSuccess) return cuda_fail(e);
    }
    return static_cast<int>(site);
#else
    (void)clear;
    return 0;
#endif
}

int attn_debug_selftest(void) {
#ifdef ATTN_DEBUG
    int sms = 0;
    int rc = device_setup(&sms);
    if (rc != ATTN_OK) return rc;
    attn::debug_selftest_kernel<<<1, 32>>>();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
#else
    return ATTN_ERR_UNSUPPORTED;
#endif
}

int attn_selftest_wait_timeout(int64_t limit_ns) {
    if (limit_ns < 1 || limit_ns > 1000000000LL) return ATTN_ERR_SHAPE;
    int sms = 0;
    int rc = device_setup(&sms);
    if (rc != ATTN_OK) return rc;
    attn::selftest_wait_kernel<<<1, 32>>>(static_cast<unsigned long long>(limit_ns));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return attn_device_error(1);
}

int attn_version(void) { return 100; }

}  // extern "C"
