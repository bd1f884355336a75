// Backward pass of the exact attention forward, on the tensor cores (sm_103a). Included
// into attn_fwd.cu inside namespace attn, so it shares the device status word, the
// bounded waits and the inline-PTX wrappers.
//
// Gradients, for the upstream gradient dO of O (the chain rule through the definition):
//   P  = exp(scale S - lse)            (the forward's softmax weights; 0 where masked)
//   dP = dO V^T,  D_i = dO_i . O_i     (D_i = sum_j P_ij dP_ij, since O_i = sum_j P_ij V_j)
//   dS = P o (dP - D)
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO   (dK, dV summed over a group's heads)
//
// Three kernels:
//   bwd_preprocess_kernel  per query row lse log2(e) and D = rowsum(dO o O) in fp32 (D / 8
//                          lanes per row, several rows per warp), each head's rows padded
//                          to a multiple of 128
//   bwd kernel, MODE 0     key-stationary: a CTA holds K_j, V_j of one key tile and
//                          streams (Q_i, dO_i) over every query head of the group and
//                          every query tile that sees the keys: S^T = K Q^T and
//                          dP^T = V dO^T into tensor memory, P^T and dS^T by the compute
//                          warps, then dV += P^T dO and dK += dS^T Q accumulate in tensor
//                          memory across the whole stream
//   bwd kernel, MODE 1     query-stationary: holds Q_i, dO_i and streams (K_j, V_j):
//                          S = Q K^T, dP = dO V^T, dS, then dQ += dS K (no atomics, so
//                          the result does not depend on the order of the key tiles)
// Each streamed 128-row tile is taken in two sub-steps of 64 rows (queries in MODE 0,
// keys in MODE 1), with two tensor-memory buffers for S and dP: the tensor core computes
// one sub-step's S and dP while the compute warps turn the other's into P and dS. The
// streamed tiles arrive in 64-row halves through a ring of half-slots, each released as
// soon as its own sub-step's products have been issued.
// Warps: 0-3 compute the first sub-step of every tile and 4-7 the second (one tensor-
// memory row each thread, so the two run side by side on one tile), 8 TMA producer, 9
// MMA issuer. Tensor memory: sub-step buffer h at [128h, 128h + 128) with S (or S^T) in
// its first 64 columns and dP in the other 64 (P and dS, bf16, over their first 32),
// then the accumulators from column 256.
#pragma once

constexpr int BWD_THREADS = 320;
constexpr int BWD_WARP_TMA = 8;
constexpr int BWD_WARP_MMA = 9;

struct BwdParams {
    const float *lse2;  // lse log2(e) per query row, fp32 [B * Hq * N_pad] (0 past N)
    const float *dsum;  // D = dO . O per query row, fp32 [B * Hq * N_pad] (0 past N)
    __nv_bfloat16 *dq, *dk, *dv;
    const int *key_len;
    int B, Hq, Hkv, N, N_pad, group;
    int causal, window, sym;
    int n_kv, num_units;
    float sl2, scale;
    unsigned long long timeout_ns;
    FastDiv div_bhkv, div_hkv, div_bhq, div_hq, div_group;
};

template <int D>
struct BwdCfg {
    static constexpr int CHUNK_BYTES = BM * 128;  // 128 rows x 64 bf16 columns, 128-byte swizzled
    static constexpr int NCHUNK = D / 64;
    static constexpr int TILE_BYTES = CHUNK_BYTES * NCHUNK;
    static constexpr int HCHUNK_BYTES = CHUNK_BYTES / 2;       // 64 rows x 64 columns
    static constexpr int HTILE_BYTES = TILE_BYTES / 2;         // 64 rows x d
    static constexpr int HSTAGES = D == 64 ? 8 : 4;            // streamed half-tile pairs in flight
    // the two stationary tiles, in FIX_BUFS buffers: with two (d = 64, where shared memory
    // has room), the producer loads the next unit's tiles while the current unit computes
    static constexpr int FIX_BUFS = D == 64 ? 2 : 1;
    static constexpr int SMEM_FIX = 0;
    static constexpr int SMEM_RING = FIX_BUFS * 2 * TILE_BYTES;  // HSTAGES x two streamed half tiles
    static constexpr int SMEM_VEC = SMEM_RING + HSTAGES * 2 * HTILE_BYTES;  // per half-slot: lse2, D
    static constexpr int VEC_BYTES = 2 * 64 * 4;
    static constexpr int SMEM_BAR = SMEM_VEC + HSTAGES * VEC_BYTES;
    static constexpr int B_FIXFULL = 0, B_FIXEMPTY = FIX_BUFS;  // FIX_BUFS each
    static constexpr int B_FULL = 2 * FIX_BUFS, B_EMPTY = B_FULL + HSTAGES;
    static constexpr int B_SDP = B_EMPTY + HSTAGES;  // 2: S and dP of sub-step h computed
    static constexpr int B_PDS = B_SDP + 2;        // 2: P (MODE 0) and dS of sub-step h written (4 warps)
    static constexpr int B_ACC = B_PDS + 2;        // 2: accumulators of a unit complete (per set)
    static constexpr int B_AFREE = B_ACC + 2;      // 2: read by the epilogue (8 warps; per set)
    static constexpr int B_DRAIN = B_AFREE + 2;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int SMEM_CTL = SMEM_BAR + NUM_BARS * 8;
    static constexpr int SMEM_ALLOC = SMEM_CTL + 16 + 1024;
    static constexpr uint32_t COL_BUF = 128;  // sub-step buffer h starts at column 128h
    static constexpr uint32_t COL_S = 0, COL_DP = 64, COL_A0 = 256, COL_A1 = 256 + D;  // set a: + a BwdAcc::COLS
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * D <= (int)TMEM_COLS, "tensor memory budget");
};

// Accumulator sets of a kernel: two where tensor memory has room beside the two sub-step
// buffers (d = 64, and the dQ kernel, whose only accumulator is dQ), so that a unit's
// products can start while the compute warps still have the previous unit's accumulators
// to read; one for dK and dV at d = 128.
template <int D, int MODE>
struct BwdAcc {
    static constexpr int BUFS = (D == 64 || MODE == 1) ? 2 : 1;
    static constexpr uint32_t COLS = MODE == 0 ? 2 * D : D;  // dV and dK, or dQ
    static_assert(256 + BUFS * COLS <= TMEM_COLS, "accumulator sets in tensor memory");
};

// Per query row of each head (N_pad rows, one warp each): lse log2(e) and
// D = sum_c dO O in fp32; rows from N to N_pad get zeros.
// Rows per warp of bwd_preprocess_kernel: a row is D / 8 lanes of 16 bytes, and each lane
// keeps PRE_LOADS rows' loads in flight before reducing.
constexpr int PRE_LOADS = 4;
template <int D>
__host__ __device__ constexpr int pre_rows_per_warp() { return PRE_LOADS * (32 / (D / 8)); }

template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16 *__restrict__ o,
                                                             const __nv_bfloat16 *__restrict__ dout,
                                                             const float *__restrict__ lse,
                                                             float *__restrict__ lse2, float *__restrict__ dsum,
                                                             long long BH, int N, int N_pad) {
    constexpr int LPR = D / 8;   // lanes per row, 8 bf16 (16 bytes) each
    constexpr int RPL = 32 / LPR;  // rows per warp-wide load
    constexpr int RPW = pre_rows_per_warp<D>();
    static_assert(BM % RPW == 0, "a warp's rows lie in one head (N_pad is a multiple of BM)");
    // the dK/dV kernel is launched as a programmatic dependent: it may be scheduled now
    // and runs its prologue, then waits for this grid before reading the row terms
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long prow0 = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * RPW;
    const int lane = threadIdx.x & 31;
    if (prow0 >= BH * N_pad) return;
    if (!ATTN_CHECK(prow0 >= 0 && N <= N_pad && N_pad % RPW == 0, 25u)) return;
    const long long h = prow0 / N_pad;
    const int i0 = static_cast<int>(prow0 - h * N_pad);
    const int sub = lane / LPR, part = lane - sub * LPR;
    // every load first, then the products: PRE_LOADS independent 16-byte loads per operand
    uint4 x[PRE_LOADS], y[PRE_LOADS];
#pragma unroll
    for (int u = 0; u < PRE_LOADS; ++u) {
        const int i = i0 + u * RPL + sub;
        if (i < N) {
            const long long off = (h * N + i) * D + part * 8;
            x[u] = __ldg(reinterpret_cast<const uint4 *>(o + off));
            y[u] = __ldg(reinterpret_cast<const uint4 *>(dout + off));
        } else {
            x[u] = make_uint4(0u, 0u, 0u, 0u);
            y[u] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    float acc[PRE_LOADS];
#pragma unroll
    for (int u = 0; u < PRE_LOADS; ++u) {
        const uint32_t xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w}, ys[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            a = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), a);
            a = fmaf(__uint_as_float(xs[e] & 0xFFFF0000u), __uint_as_float(ys[e] & 0xFFFF0000u), a);
        }
        // sum over the LPR lanes of the row (aligned groups of LPR lanes)
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
        acc[u] = a;
    }
    if (part == 0) {
#pragma unroll
        for (int u = 0; u < PRE_LOADS; ++u) {
            const int i = i0 + u * RPL + sub;
            const long long prow = prow0 + u * RPL + sub;
            lse2[prow] = i < N ? __ldg(lse + h * N + i) * 1.4426950408889634f : 0.f;
            dsum[prow] = i < N ? acc[u] : 0.f;
        }
    }
}

__device__ __forceinline__ int bwd_valid_len(const BwdParams &p, int b) {
    if (!p.key_len) return p.N;
    return min(max(__ldg(p.key_len + b), 0), p.N);
}

// Queries a key row k (of a batch with valid length L) is visible to: [qlo, qhi], empty
// when qlo > qhi. (The transpose of the forward's key interval of a query row.)
__device__ __forceinline__ void key_query_interval(const BwdParams &p, int k, int L, int &qlo, int &qhi) {
    qlo = 0;
    qhi = L - 1;
    if (k >= L) {
        qlo = 1;
        qhi = 0;
        return;
    }
    if (p.causal) qlo = k;
    if (p.window > 0) {
        qhi = min(qhi, k + p.window - 1);
        if (p.sym) qlo = max(qlo, k - p.window + 1);
    }
}

// Keys a query row q is visible to: [klo, khi] (as in the forward).
__device__ __forceinline__ void query_key_interval(const BwdParams &p, int q, int L, int &klo, int &khi) {
    klo = 0;
    khi = L - 1;
    if (q >= L) {
        klo = 1;
        khi = 0;
        return;
    }
    if (p.causal) khi = min(khi, q);
    if (p.sym) khi = min(khi, q + p.window - 1);
    if (p.window > 0) klo = max(0, q - p.window + 1);
}

// What one unit covers. MODE 0: the key tile j of (b, hkv) and the range of query tiles
// [lo, hi) every head of the group streams. MODE 1: the query tile i of (b, hq) and the
// key tiles [lo, hi) it streams.
struct BwdUnit {
    int b, tile, zfix, zstream0, L, lo, hi, steps;
};

template <int MODE>
__device__ __forceinline__ BwdUnit bwd_unit(int u, const BwdParams &p) {
    BwdUnit w;
    if constexpr (MODE == 0) {
        const int BHkv = p.B * p.Hkv;
        const int pr = fdiv(u, p.div_bhkv);
        const int bhkv = u - pr * BHkv;
        w.b = fdiv(bhkv, p.div_hkv);
        const int hkv = bhkv - w.b * p.Hkv;
        // heaviest first: under the look-ahead mask key tile 0 is seen by every query tile
        w.tile = pr;
        w.zfix = bhkv;
        w.zstream0 = w.b * p.Hq + hkv * p.group;  // first query head of the group
        w.L = bwd_valid_len(p, w.b);
        w.lo = w.hi = 0;
        const int k0 = w.tile * BN;
        if (k0 < w.L) {
            int qlo0, qhi0, qlo1, qhi1;
            key_query_interval(p, k0, w.L, qlo0, qhi0);
            key_query_interval(p, min(w.L, k0 + BN) - 1, w.L, qlo1, qhi1);
            const int qlo = qlo0, qhi = max(qhi0, qhi1);
            if (qlo <= qhi) {
                w.lo = qlo / BM;
                w.hi = qhi / BM + 1;
            }
        }
        w.steps = p.group * (w.hi - w.lo);
    } else {
        const int BHq = p.B * p.Hq;
        const int pr = fdiv(u, p.div_bhq);
        const int bh = u - pr * BHq;
        w.b = fdiv(bh, p.div_hq);
        const int hq = bh - w.b * p.Hq;
        w.tile = p.n_kv - 1 - pr;  // heaviest first under the look-ahead mask
        w.zfix = bh;
        w.zstream0 = w.b * p.Hkv + fdiv(hq, p.div_group);
        w.L = bwd_valid_len(p, w.b);
        w.lo = w.hi = 0;
        const int q0 = w.tile * BM;
        if (q0 < w.L) {
            int klo0, khi0, klo1, khi1;
            query_key_interval(p, q0, w.L, klo0, khi0);
            query_key_interval(p, min(w.L, q0 + BM) - 1, w.L, klo1, khi1);
            const int klo = klo0, khi = max(khi0, khi1);
            if (klo <= khi) {
                w.lo = klo / BN;
                w.hi = khi / BN + 1;
            }
        }
        w.steps = w.hi - w.lo;
    }
    return w;
}

// tm_fix0, tm_fix1: the stationary operands in 128-row boxes (MODE 0: K, V; MODE 1: Q,
// dO); tm_str0, tm_str1: the streamed ones in 64-row boxes (MODE 0: Q, dO; MODE 1: K, V)
template <int D, int MODE>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_fix0, const __grid_constant__ CUtensorMap tm_fix1,
                    const __grid_constant__ CUtensorMap tm_str0, const __grid_constant__ CUtensorMap tm_str1,
                    const BwdParams p) {
    using C = BwdCfg<D>;
    using A = BwdAcc<D, MODE>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + C::SMEM_CTL);
    auto bar = [&](int i) -> uint32_t { return sb + C::SMEM_BAR + 8u * static_cast<uint32_t>(i); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < C::FIX_BUFS; ++b) {
            ptx::mbar_init(bar(C::B_FIXFULL + b), 1);
            ptx::mbar_init(bar(C::B_FIXEMPTY + b), 1);
        }
        for (int s = 0; s < C::HSTAGES; ++s) {
            ptx::mbar_init(bar(C::B_FULL + s), 1);
            ptx::mbar_init(bar(C::B_EMPTY + s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            ptx::mbar_init(bar(C::B_SDP + h), 1);
            ptx::mbar_init(bar(C::B_PDS + h), 4);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bar(C::B_ACC + a), 1);
            ptx::mbar_init(bar(C::B_AFREE + a), 8);
        }
        ptx::mbar_init(bar(C::B_DRAIN), 1);
        ctl->abort = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == BWD_WARP_TMA && lane == 0) {
        ptx::prefetch_tensormap(&tm_fix0);
        ptx::prefetch_tensormap(&tm_fix1);
        ptx::prefetch_tensormap(&tm_str0);
        ptx::prefetch_tensormap(&tm_str1);
    }
    if (warp == BWD_WARP_MMA) {
        ptx::tmem_alloc(sb + C::SMEM_CTL, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    // Programmatic dependent launch: the prologue above may overlap the previous kernel
    // of the pass; every read of the row terms (and of the inputs) comes after this wait
    // for it to complete. The next kernel (dQ after dK/dV) may then be scheduled: it
    // takes an SM as each CTA of this one exits.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    volatile uint32_t *abort_flag = &ctl->abort;
    const unsigned long long limit = p.timeout_ns;
    // half-slot n of the ring: streamed operand 0 at half_base(n), operand 1 HTILE_BYTES on
    auto half_base = [&](uint32_t slot) -> uint32_t { return sb + C::SMEM_RING + slot * 2 * C::HTILE_BYTES; };

    if (warp == BWD_WARP_TMA) {
        // ================================================================ producer
        uint32_t hit = 0, fix_it = 0;
        bool ok = true;
        for (int kk = 0, u = snake_unit(0); ok && u < p.num_units; u = snake_unit(++kk)) {
            const BwdUnit w = bwd_unit<MODE>(u, p);
            if (w.steps == 0) continue;
            const uint32_t fb = fix_it % C::FIX_BUFS;
            ok = wait_warp(bar(C::B_FIXEMPTY + fb), ((fix_it / C::FIX_BUFS) & 1u) ^ 1u, abort_flag, limit);
            ++fix_it;
            if (!ok) break;
            const uint32_t fdst = sb + C::SMEM_FIX + fb * 2 * C::TILE_BYTES;
            // debug build: the stationary tile's head and rows
            if (!ATTN_CHECK(w.zfix >= 0 && w.zfix < p.B * (MODE == 0 ? p.Hkv : p.Hq) && w.tile >= 0 &&
                                w.tile * BM < p.N,
                            20u))
                continue;
            ptx::mbar_arrive_expect_tx_elect(bar(C::B_FIXFULL + fb), 2 * C::TILE_BYTES);
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c) {
                ptx::tma_load_3d_elect(fdst + c * C::CHUNK_BYTES, &tm_fix0, bar(C::B_FIXFULL + fb), c * 64,
                                       w.tile * BM, w.zfix);
                ptx::tma_load_3d_elect(fdst + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_fix1, bar(C::B_FIXFULL + fb),
                                       c * 64, w.tile * BM, w.zfix);
            }
            for (int s = 0; ok && s < w.steps; ++s) {
                // MODE 0: step s = (head g of the group, query tile t); MODE 1: key tile t
                const int n_t = w.hi - w.lo;
                const int g = MODE == 0 ? s / n_t : 0;
                const int t = w.lo + (MODE == 0 ? s - g * n_t : s);
                const int zs = w.zstream0 + g;
                for (int h = 0; ok && h < 2; ++h) {
                    const uint32_t slot = hit % C::HSTAGES, ph = ((hit / C::HSTAGES) & 1u) ^ 1u;
                    ok = wait_warp(bar(C::B_EMPTY + slot), ph, abort_flag, limit);
                    if (!ok) break;
                    ++hit;
                    const uint32_t dst = half_base(slot);
                    const int row0 = t * BM + 64 * h;
                    // debug build: the ring half-slot, the streamed head and rows (and, for
                    // dK/dV, the row terms read beside them)
                    if (!ATTN_CHECK(slot < static_cast<uint32_t>(C::HSTAGES) && zs >= 0 &&
                                        zs < p.B * (MODE == 0 ? p.Hq : p.Hkv) && row0 >= 0 && row0 + 64 <= p.N_pad,
                                    21u))
                        continue;
                    if constexpr (MODE == 0) {
                        // the half tile's 64 values of lse log2(e) and of D land beside it
                        const uint32_t vec = sb + C::SMEM_VEC + slot * C::VEC_BYTES;
                        const size_t idx = static_cast<size_t>(zs) * p.N_pad + row0;
                        ptx::mbar_arrive_expect_tx_elect(bar(C::B_FULL + slot), 2 * C::HTILE_BYTES + C::VEC_BYTES);
                        ptx::bulk_load_elect(vec, p.lse2 + idx, 64 * 4, bar(C::B_FULL + slot));
                        ptx::bulk_load_elect(vec + 64 * 4, p.dsum + idx, 64 * 4, bar(C::B_FULL + slot));
                    } else {
                        ptx::mbar_arrive_expect_tx_elect(bar(C::B_FULL + slot), 2 * C::HTILE_BYTES);
                    }
#pragma unroll
                    for (int c = 0; c < C::NCHUNK; ++c) {
                        ptx::tma_load_3d_elect(dst + c * C::HCHUNK_BYTES, &tm_str0, bar(C::B_FULL + slot), c * 64,
                                               row0, zs);
                        ptx::tma_load_3d_elect(dst + C::HTILE_BYTES + c * C::HCHUNK_BYTES, &tm_str1,
                                               bar(C::B_FULL + slot), c * 64, row0, zs);
                    }
                }
            }
        }
        if (!ok) {
            for (uint32_t slot = 0; slot < static_cast<uint32_t>(C::HSTAGES); ++slot) {
                if (hit <= slot) continue;
                const uint32_t last = (hit - 1u - slot) / C::HSTAGES * C::HSTAGES + slot;
                drain_wait(bar(C::B_FULL + slot), (last / C::HSTAGES) & 1u, 100000000ull);
            }
            for (uint32_t b = 0; b < static_cast<uint32_t>(C::FIX_BUFS); ++b) {
                const uint32_t n_b = (fix_it + C::FIX_BUFS - 1u - b) / C::FIX_BUFS;  // loads into buffer b
                if (n_b) drain_wait(bar(C::B_FIXFULL + b), (n_b - 1u) & 1u, 100000000ull);
            }
        }
    } else if (warp == BWD_WARP_MMA) {
        // ================================================================ MMA issuer
        // All 32 lanes run this loop with identical values; each MMA and commit is
        // issued by one elected lane. MMAs of one thread run in issue order, so a product
        // may overwrite tensor-memory columns that earlier products read.
        constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(BM, 64, false);
        constexpr uint32_t IDESC_ACC = ptx::idesc_bf16_f32(BM, D, true);
        uint32_t hit = 0, fix_use = 0, pds_use0 = 0, pds_use1 = 0, acc_fills = 0;
        bool ok = true;
        // sub-step h: S (S^T) and dP (dP^T) = A B^T over d, both operands K-major: A the
        // stationary 128-row tile, B the streamed 64-row half tile
        auto issue_sdp = [&](int h, uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1) {
            const uint32_t col = C::COL_BUF * h;
            // debug build: S and dP of the sub-step inside tensor memory
            if (!ATTN_CHECK(col + C::COL_DP + 64 <= TMEM_COLS && col + C::COL_S + 64 <= TMEM_COLS, 22u)) return;
            const uint64_t a0d = ptx::sdesc_sw128(a0, 16, 1024), a1d = ptx::sdesc_sw128(a1, 16, 1024);
            const uint64_t b0d = ptx::sdesc_sw128(b0, 16, 1024), b1d = ptx::sdesc_sw128(b1, 16, 1024);
            // four K steps of 32 bytes per 128-byte swizzled slab, one asm statement each
#pragma unroll
            for (int g = 0; g < D / 64; ++g) {
                const uint64_t aoff = static_cast<uint64_t>(g * C::CHUNK_BYTES) >> 4;
                const uint64_t boff = static_cast<uint64_t>(g * C::HCHUNK_BYTES) >> 4;
                ptx::mma_ss4_elect<2>(tmem + col + C::COL_S, a0d + aoff, b0d + boff, IDESC_S, g > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int g = 0; g < D / 64; ++g) {
                const uint64_t aoff = static_cast<uint64_t>(g * C::CHUNK_BYTES) >> 4;
                const uint64_t boff = static_cast<uint64_t>(g * C::HCHUNK_BYTES) >> 4;
                ptx::mma_ss4_elect<2>(tmem + col + C::COL_DP, a1d + aoff, b1d + boff, IDESC_S, g > 0 ? 1u : 0u);
            }
            ptx::mma_commit_elect(bar(C::B_SDP + h));
        };
        // D[tmem] (+)= A[tmem, bf16] B for one sub-step: A = 64 rows' worth of P / dS (32
        // packed columns), B = a streamed [64 x d] half tile read MN-major
        auto issue_acc = [&](uint32_t col_d, uint32_t col_a, uint32_t b_addr, bool accumulate) {
            // debug build: the accumulator and the packed A operand inside tensor memory
            if (!ATTN_CHECK(col_d + D <= TMEM_COLS && col_a + 32 <= TMEM_COLS, 23u)) return;
            const uint64_t bd = ptx::sdesc_sw128(b_addr, C::HCHUNK_BYTES, 1024);
            // four K steps of 16 rows (8 packed columns of A, 2048 bytes of B) in one asm statement
            ptx::mma_ts4_elect<8, 128>(tmem + col_d, tmem + col_a, bd, IDESC_ACC, accumulate ? 1u : 0u);
        };
        // the accumulating products of sub-step h (half tile at hb), once the compute warps
        // wrote its P / dS
        auto issue_products = [&](int h, uint32_t hb, bool accumulate, uint32_t acol) -> bool {
            uint32_t &use = h ? pds_use1 : pds_use0;
            if (!wait_warp(bar(C::B_PDS + h), use & 1u, abort_flag, limit)) return false;
            ++use;
            ptx::tc_fence_after();
            const uint32_t buf = C::COL_BUF * h;
            if constexpr (MODE == 0) {
                issue_acc(C::COL_A0 + acol, buf + C::COL_S, hb + C::HTILE_BYTES, accumulate);  // dV += P^T dO
                issue_acc(C::COL_A1 + acol, buf + C::COL_DP, hb, accumulate);                 // dK += dS^T Q
            } else {
                issue_acc(C::COL_A0 + acol, buf + C::COL_S, hb, accumulate);                  // dQ += dS K
            }
            return true;
        };
        auto next_half = [&](uint32_t &slot) -> bool {
            slot = hit % C::HSTAGES;
            const uint32_t ph = (hit / C::HSTAGES) & 1u;
            ++hit;
            if (!wait_warp(bar(C::B_FULL + slot), ph, abort_flag, limit)) return false;
            ptx::tc_fence_after();
            return true;
        };
        for (int kk = 0, u = snake_unit(0); ok && u < p.num_units; u = snake_unit(++kk)) {
            const BwdUnit w = bwd_unit<MODE>(u, p);
            if (w.steps == 0) continue;
            const uint32_t fb = fix_use % C::FIX_BUFS;
            ok = wait_warp(bar(C::B_FIXFULL + fb), (fix_use / C::FIX_BUFS) & 1u, abort_flag, limit);
            ++fix_use;
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t f0 = sb + C::SMEM_FIX + fb * 2 * C::TILE_BYTES, f1 = f0 + C::TILE_BYTES;
            // this unit's accumulator set (units alternate between the sets)
            const uint32_t aset = acc_fills % A::BUFS, aph = (acc_fills / A::BUFS) & 1u;
            const uint32_t acol = aset * A::COLS;
            ++acc_fills;
            uint32_t prev_slot = 0;
            for (int s = 0; s < w.steps; ++s) {
                // order: S, dP of (s, 0); products of (s - 1, 1); S, dP of (s, 1); products
                // of (s, 0). Buffer h is rewritten only after the products that read its P
                // and dS were issued, and the tensor core always has the next sub-step's
                // S and dP to compute while the compute warps work. A half-slot is
                // released right after its sub-step's products.
                uint32_t slot0, slot1;
                if (!(ok = next_half(slot0))) break;
                issue_sdp(0, f0, f1, half_base(slot0), half_base(slot0) + C::HTILE_BYTES);
                if (s > 0) {
                    if (!(ok = issue_products(1, half_base(prev_slot), true, acol))) break;
                    ptx::mma_commit_elect(bar(C::B_EMPTY + prev_slot));
                }
                if (!(ok = next_half(slot1))) break;
                issue_sdp(1, f0, f1, half_base(slot1), half_base(slot1) + C::HTILE_BYTES);
                if (s == 0) {
                    // the unit's first products overwrite its accumulator set: both compute
                    // warpgroups must have read what the unit ACC_BUFS back left there (a
                    // fresh barrier passes parity 1)
                    ok = wait_warp(bar(C::B_AFREE + aset), aph ^ 1u, abort_flag, limit);
                    if (!ok) break;
                    ptx::tc_fence_after();
                }
                if (!(ok = issue_products(0, half_base(slot0), s > 0, acol))) break;
                ptx::mma_commit_elect(bar(C::B_EMPTY + slot0));
                prev_slot = slot1;
            }
            if (!ok) break;
            if (!(ok = issue_products(1, half_base(prev_slot), true, acol))) break;
            ptx::mma_commit_elect(bar(C::B_EMPTY + prev_slot));
            ptx::mma_commit_elect(bar(C::B_FIXEMPTY + fb));
            ptx::mma_commit_elect(bar(C::B_ACC + aset));
        }
        ptx::mma_commit_elect(bar(C::B_DRAIN));
        drain_wait(bar(C::B_DRAIN), 0u, 100000000ull);
        __syncwarp();
    } else if (warp < 8) {
        // ================================================================ compute
        // warpgroup h (warps 4h .. 4h + 3) takes sub-step h of every tile
        const int h = warp >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t t_s = tmem + lane_off + C::COL_BUF * h + C::COL_S;
        const uint32_t t_dp = tmem + lane_off + C::COL_BUF * h + C::COL_DP;
        uint32_t hit = 0, sdp_use = 0, acc_use = 0;
        bool ok = true;
        // Epilogue of a unit, split between the warpgroups: MODE 0 writes dV (warpgroup 0)
        // and scale * dK (warpgroup 1) of the key rows; MODE 1 writes scale * dQ, columns
        // [0, d/2) from warpgroup 0 and [d/2, d) from warpgroup 1. `fill` is the unit's
        // index among those with something to stream (its accumulator set and phase); a
        // unit with nothing to stream writes zeros.
        auto epilogue = [&](int zfix, int r_row, bool has, uint32_t fill) -> bool {
            const uint32_t aset = fill % A::BUFS;
            if (has) {
                if (!wait_warp(bar(C::B_ACC + aset), (fill / A::BUFS) & 1u, abort_flag, limit)) return false;
                ptx::tc_fence_after();
            }
            __nv_bfloat16 *out = MODE == 0 ? (h == 0 ? p.dv : p.dk) : p.dq;
            const float mul = (MODE == 0 && h == 0) ? 1.f : p.scale;
            constexpr int NC = MODE == 0 ? D / 32 : D / 64;  // 32-column chunks this warpgroup writes
            const int col0 = MODE == 0 ? 0 : h * (D / 2);
            const uint32_t t_acc = tmem + lane_off + (MODE == 0 ? (h == 0 ? C::COL_A0 : C::COL_A1) : C::COL_A0) +
                                   aset * A::COLS + col0;
#pragma unroll 1
            for (int c = 0; c < NC; ++c) {
                uint32_t r[32];
                if (has) {
                    ptx::tmem_ld32(t_acc + 32 * c, r);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = 0u;
                }
                // debug build: the gradient row inside its output
                if (r_row < p.N && ATTN_CHECK(zfix >= 0 && zfix < p.B * (MODE == 0 ? p.Hkv : p.Hq), 24u)) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + (static_cast<size_t>(zfix) * p.N + r_row) * D + col0 +
                                                           32 * c);
#pragma unroll
                    for (int g4 = 0; g4 < 4; ++g4) {
                        uint4 val;
                        val.x = ptx::pack_bf16x2(__uint_as_float(r[8 * g4 + 0]) * mul,
                                                 __uint_as_float(r[8 * g4 + 1]) * mul);
                        val.y = ptx::pack_bf16x2(__uint_as_float(r[8 * g4 + 2]) * mul,
                                                 __uint_as_float(r[8 * g4 + 3]) * mul);
                        val.z = ptx::pack_bf16x2(__uint_as_float(r[8 * g4 + 4]) * mul,
                                                 __uint_as_float(r[8 * g4 + 5]) * mul);
                        val.w = ptx::pack_bf16x2(__uint_as_float(r[8 * g4 + 6]) * mul,
                                                 __uint_as_float(r[8 * g4 + 7]) * mul);
                        dst[g4] = val;
                    }
                }
            }
            if (has) {
                // the accumulators are read: a later unit's first products may overwrite them
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(C::B_AFREE + aset));
            }
            return true;
        };
        // With two accumulator sets a unit's epilogue waits until this warpgroup has done
        // its first sub-step of the next unit: the unit's last products then complete
        // while the warps compute, instead of while they wait.
        bool pend = false;
        int pend_zfix = 0, pend_row = 0;
        uint32_t pend_fill = 0;
        for (int kk = 0, u = snake_unit(0); ok && u < p.num_units; u = snake_unit(++kk)) {
            const BwdUnit w = bwd_unit<MODE>(u, p);
            const int r_abs = w.tile * BM + row;  // this thread's key (MODE 0) or query (MODE 1)
            // MODE 1: the row's lse (log2 units) and D
            float row_lse2 = 0.f, row_d = 0.f;
            if constexpr (MODE == 1) {
                if (r_abs < p.N) {
                    const size_t idx = static_cast<size_t>(w.zfix) * p.N_pad + r_abs;
                    row_lse2 = __ldg(p.lse2 + idx);
                    row_d = __ldg(p.dsum + idx);
                }
            }
            int ilo, ihi;  // this row's visible column interval (absolute positions)
            if constexpr (MODE == 0)
                key_query_interval(p, r_abs, w.L, ilo, ihi);
            else
                query_key_interval(p, r_abs, w.L, ilo, ihi);
            for (int s = 0; ok && s < w.steps; ++s) {
                const int n_t = w.hi - w.lo;
                const int g = MODE == 0 ? s / n_t : 0;
                const int t = w.lo + (MODE == 0 ? s - g * n_t : s);
                (void)g;
                // half-slot of this sub-step: the tile's two halves take consecutive slots
                const uint32_t slot = (hit + h) % C::HSTAGES, ph = ((hit + h) / C::HSTAGES) & 1u;
                hit += 2;
                const float *vec = reinterpret_cast<const float *>(smem + C::SMEM_VEC + slot * C::VEC_BYTES);
                if constexpr (MODE == 0) {
                    // the half tile's lse and D were staged with it
                    ok = wait_warp(bar(C::B_FULL + slot), ph, abort_flag, limit);
                    if (!ok) break;
                }
                // columns 64h .. 64h + 63 of the tile; those this row sees: [c_lo, c_hi]
                const int c0 = t * BN;
                const int c_hi = min(ihi, c0 + BN - 1) - c0;
                const int c_lo = max(ilo, c0) - c0;
                const bool none = c_hi < c_lo;
                const uint32_t span = none ? 0u : static_cast<uint32_t>(c_hi - c_lo);
                const uint32_t base = none ? 0xFFFFFFFFu : static_cast<uint32_t>(c_lo);
                const bool covers = !none && c_lo <= 64 * h && c_hi >= 64 * h + 63;
                const bool need_mask = !__all_sync(0xffffffffu, covers);
                ok = wait_warp(bar(C::B_SDP + h), sdp_use & 1u, abort_flag, limit);
                ++sdp_use;
                if (!ok) break;
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t sr[32], dr[32];
                    ptx::tmem_ld32(t_s + 32 * c, sr);
                    ptx::tmem_ld32(t_dp + 32 * c, dr);
                    const int cb = 64 * h + 32 * c;  // first column of the chunk in the tile
                    ptx::tmem_wait_ld();
                    uint32_t pk[16], dk16[16];
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        float4 l4, d4;
                        if constexpr (MODE == 0) {
                            l4 = *reinterpret_cast<const float4 *>(vec + 32 * c + 4 * e4);
                            d4 = *reinterpret_cast<const float4 *>(vec + 64 + 32 * c + 4 * e4);
                        } else {
                            l4 = make_float4(row_lse2, row_lse2, row_lse2, row_lse2);
                            d4 = make_float4(row_d, row_d, row_d, row_d);
                        }
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
                        float pp[4], ds[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int e = 4 * e4 + q;
                            float pv = ptx::ex2(fmaf(__uint_as_float(sr[e]), p.sl2, -lv[q]));
                            if (need_mask && static_cast<uint32_t>(cb + e) - base > span) pv = 0.f;
                            pp[q] = pv;
                            ds[q] = pv * (__uint_as_float(dr[e]) - dv[q]);
                        }
                        pk[2 * e4] = ptx::pack_bf16x2(pp[0], pp[1]);
                        pk[2 * e4 + 1] = ptx::pack_bf16x2(pp[2], pp[3]);
                        dk16[2 * e4] = ptx::pack_bf16x2(ds[0], ds[1]);
                        dk16[2 * e4 + 1] = ptx::pack_bf16x2(ds[2], ds[3]);
                    }
                    if constexpr (MODE == 0) {
                        ptx::tmem_st16(t_s + 16 * c, pk);     // P^T, A of dV += P^T dO
                        ptx::tmem_st16(t_dp + 16 * c, dk16);  // dS^T, A of dK += dS^T Q
                    } else {
                        ptx::tmem_st16(t_s + 16 * c, dk16);   // dS, A of dQ += dS K
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(C::B_PDS + h));
                if (A::BUFS > 1 && pend) {
                    pend = false;
                    if (!(ok = epilogue(pend_zfix, pend_row, true, pend_fill))) break;
                }
            }
            if (!ok) break;
            const bool has = w.steps > 0;
            if (A::BUFS > 1 && pend) {
                // (a unit with nothing to stream: the previous unit's epilogue first)
                pend = false;
                if (!(ok = epilogue(pend_zfix, pend_row, true, pend_fill))) break;
            }
            const uint32_t fill = has ? acc_use++ : 0u;
            if (has && A::BUFS > 1) {
                pend = true;
                pend_zfix = w.zfix;
                pend_row = r_abs;
                pend_fill = fill;
            } else if (!(ok = epilogue(w.zfix, r_abs, has, fill))) {
                break;
            }
        }
        if (A::BUFS > 1 && ok && pend) ok = epilogue(pend_zfix, pend_row, true, pend_fill);
        (void)ok;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == BWD_WARP_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}
