// Sparse GQA attention on the 5th-generation tensor cores, for 16-bit K/V
// caches with dk = dv = 128 and up to 16 query heads per kv head (the
// block-pooled decode's attention, "QSA" commit message, llama.cpp commit
// c88c916636; the gathered decode, "Gather OpenPangu DSA decode reads",
// ik_llama_opt commit log):
//     l[h, j] = scale * q[r, h] . K[j, g], p = softmax_j(l),
//     out[r, h] = sum_j p[h, j] V[j, g]      for j in the row's selection.
// A query row has only G = Hq / Hkv heads per kv head (8 on the block-pooled
// decode), too few to be the M side of an MMA, so the keys are: per tile of
// 128 selected keys
//     S^T[128 keys x 16] = K_tile[128 x 128] . Q^T[128 x 16]   (M=128, N=16)
// (the G heads padded to 16 with zero rows of Q) goes to one of two TMEM
// buffers, four softmax warps (thread = key = TMEM lane) turn it into
// P = 2^(S*scale*log2e - m) with a per-head running maximum kept across the
// warps in shared memory, and write P^T (16 heads x 128 keys, bf16 or f16) as a
// K-major operand; then
//     O^T[128 dims x 16] += V_tile^T . P^T                       (M=128, N=16)
// reads V as an MN-major operand straight from the gathered tile.  A head's O
// column is rescaled in TMEM only when its maximum rises by more than 2^8.
// One CTA per (query row, kv head, key split), 12 warps: warp 0 issues the
// MMAs (QK^T of tile t+1 before PV of tile t), warps 4..7 run the softmax and
// the output, the other seven gather each tile's K and V rows with 16-byte
// cp.async copies into the 128-byte swizzle (3 stages of 64 KB).  Splits are
// merged by the CUDA-core path's combine kernel.  Every wait is bounded; a
// timeout records IDX_ERR_TIMEOUT and the CTA winds down.
#include "lidx_internal.cuh"
#include "sm100_ptx.cuh"

namespace lidx {
namespace {
using namespace sm100;

constexpr int kD = 128;                       // dk = dv
constexpr int kKeys = 128;                    // keys per tile
constexpr int kN = 16;                        // query heads per kv head, padded
constexpr int kStages = 3;
constexpr int kBlock = kKeys * 128;           // one 64-column block of a K or V tile (16 KB)
constexpr int kTile = 4 * kBlock;             // K (2 blocks) then V (2 blocks): 64 KB
constexpr int kQOff = kStages * kTile;        // Q^T operand: 2 blocks of 16 rows x 128 B
constexpr int kPOff = kQOff + 2 * kN * 128;   // two P^T tiles, each 2 blocks of 16 rows x 128 B
constexpr int kPBytes = 2 * kN * 128;
constexpr int kMaxKps = 2048;                 // selected keys per split, at most
constexpr int kRowsOff = kPOff + 2 * kPBytes;
constexpr int kWarps = 12;
constexpr int kThreads = 32 * kWarps;
constexpr int kProducerWarps = 7;             // warps 1..3 and 8..11
constexpr int kTmemCols = 64;                 // S^T buffers at 0 and 16, O^T at 32
constexpr uint32_t kOCol = 32;
constexpr float kRescaleLog2 = 8.f;

struct Ctl {
    uint64_t xfull[kStages];
    uint64_t xempty[kStages];
    uint64_t sfull[2];
    uint64_t sempty[2];
    uint64_t pready[2];
    uint64_t pvdone[2];
    uint64_t rfull[2];            // the four softmax warps' flags of a tile are in over[t & 1]
    uint64_t mfull;               // ... and, when some flag is set, their maxima in red[t & 1]
    uint64_t lfull;               // ... and their row sums in lred
    uint64_t done;
    uint8_t over[2][4];           // per warp: a key of the tile lifts a head past the rescale margin
    float red[2][4][kN];          // per-warp maxima of a tile (two tiles in turn)
    float lred[4][kN];            // per-warp row sums at the end
    float xo[kN][kD];             // split pairs, rank 0: rank 1's unnormalised output ...
    float xml[kN][2];             // ... and its maximum (natural-log units) and sum per head
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kSmemBytes = 1024 + (size_t)kRowsOff + kMaxKps * 4 + kMaxKps / 8 + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ void abort_cta(Ctl& c, int* status) {
    *(volatile int*)&c.abort = 1;
    flag(status, IDX_ERR_TIMEOUT);
}
__device__ __forceinline__ bool warp_aborted(Ctl& c) { return __any_sync(0xffffffffu, *(volatile int*)&c.abort != 0); }

__device__ __forceinline__ void st_shared_u16(uint8_t* p, uint16_t v) {
    *reinterpret_cast<uint16_t*>(p) = v;
}

template <typename T> __device__ __forceinline__ uint16_t to_bits(float x);
template <> __device__ __forceinline__ uint16_t to_bits<__nv_bfloat16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <> __device__ __forceinline__ uint16_t to_bits<__half>(float x) { return __half_as_ushort(__float2half_rn(x)); }

// the two key splits of a (row, kv head) as a cluster pair: rank 1 hands its unnormalised output,
// maximum and sum to rank 0 over DSMEM and rank 0 merges them (the combine's arithmetic)
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

template <typename T, bool kPair>
__global__ void __launch_bounds__(kThreads, 1) attn_gqa_tc_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, int64_t kv_row_stride,
    int64_t v_row_stride, int64_t kv_rows, Geom g, const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel,
    int Hq, int Hkv, float scale_log2, int splits, int kps, void* __restrict__ out, int out_dtype,
    float* __restrict__ part_o, float* __restrict__ part_ml) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qs = smem + kQOff;
    uint8_t* ps = smem + kPOff;
    int32_t* rows_s = reinterpret_cast<int32_t*>(smem + kRowsOff);
    uint32_t* vmask = reinterpret_cast<uint32_t*>(rows_s + kMaxKps);
    Ctl& c = *reinterpret_cast<Ctl*>(vmask + kMaxKps / 32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t unit = blockIdx.x;
    const int split = (int)(unit % splits);
    if (kPair) cluster_arrive_relaxed();   // (phase 0: this CTA has started)
    const int64_t rg = unit / splits;
    const int gkv = (int)(rg % Hkv);
    const int64_t r = rg / Hkv;
    const int G = Hq / Hkv;
    const int h0 = gkv * G;                        // first query head of this kv head
    const int b = (int)(r / g.T);
    const int n_kv_b = seq_n_kv(g, b);
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&c.xfull[i], 32 * kProducerWarps);
            mbar_init(&c.xempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&c.sfull[i], 1);
            mbar_init(&c.sempty[i], 4);
            mbar_init(&c.pready[i], 4);
            mbar_init(&c.pvdone[i], 1);
            mbar_init(&c.rfull[i], 4);
        }
        mbar_init(&c.mfull, 4);
        mbar_init(&c.lfull, 4);
        mbar_init(&c.done, 1);
        c.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&c.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // Q^T operand: row h = query head h0 + h (zero for h >= G), 128 dims in two 64-column blocks
    for (int i = threadIdx.x; i < kN * 16; i += kThreads) {
        const int h = i >> 4, cc = i & 15;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (h < G) x = *reinterpret_cast<const uint4*>(q + (r * Hq + h0 + h) * (int64_t)kD + cc * 8);
        *reinterpret_cast<uint4*>(qs + (cc >> 3) * (kN * 128) + h * 128 + (((cc & 7) ^ (h & 7)) << 4)) = x;
    }
    // P^T rows of padded heads stay zero
    for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(ps)[i] = make_uint4(0u, 0u, 0u, 0u);
    pdl_wait();
    // the split's selected keys -> cache rows (an in-bounds row for padding) + validity bits
    int ns = n_sel[r];
    if (ns < 0 || ns > idx_row_stride) {
        if (threadIdx.x == 0) flag(g.status, IDX_ERR_DEVICE_BOUNDS);
        ns = ns < 0 ? 0 : (int)idx_row_stride;
    }
    const int k0 = split * kps, k1 = min(ns, k0 + kps);
    const int n_tiles = k1 > k0 ? (k1 - k0 + kKeys - 1) / kKeys : 0;
    int64_t fallback = g.page_table ? 0 : seq_row0(g, b);
    if (fallback < 0) fallback = 0;
    if (fallback >= kv_rows) fallback = kv_rows - 1;
    for (int w0 = warp; w0 < n_tiles * (kKeys / 32); w0 += kWarps) {
        const int j = k0 + w0 * 32 + lane;
        bool valid = false;
        int64_t row = fallback;
        if (j < k1) {
            const int pos = idx[r * idx_row_stride + j];
            const int64_t rr = (pos >= 0 && pos < n_kv_b) ? key_row(g, b, pos) : -1;
            if (rr >= 0 && rr < kv_rows) {
                valid = true;
                row = rr;
            } else {
                flag(g.status, IDX_ERR_DEVICE_BOUNDS);
            }
        }
        rows_s[w0 * 32 + lane] = (int32_t)row;
        const uint32_t bits = __ballot_sync(0xffffffffu, valid);
        if (lane == 0) vmask[w0] = bits;
    }
    fence_proxy_async_smem();   // Q^T and the zeroed P^T (generic stores) before the MMAs read them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;

    const int producer = (warp >= 1 && warp <= 3) ? warp - 1 : (warp >= 8 ? warp - 5 : -1);
    if (producer >= 0) {
        // ------------------------------------------------------------------ gathers: a tile's K rows
        // (kv head gkv, 256 B each) then its V rows, 16 bytes per copy, 128-byte swizzle
        const char* kb = reinterpret_cast<const char*>(k) + (int64_t)gkv * kD * 2;
        const char* vb = reinterpret_cast<const char*>(v) + (int64_t)gkv * kD * 2;
        for (int t = 0; t < n_tiles; ++t) {
            const int stage = t % kStages;
            if (warp_aborted(c) || !warp_wait(&c.xempty[stage], (uint32_t)((t / kStages) & 1) ^ 1)) {
                abort_cta(c, g.status);
                break;
            }
            const uint32_t dst0 = smem_u32(smem + (size_t)stage * kTile);
            const int32_t* rr = rows_s + t * kKeys;
#pragma unroll 4
            for (int i = producer * 32 + lane; i < 2 * kKeys * 16; i += 32 * kProducerWarps) {
                const bool isv = i >= kKeys * 16;
                const int e = isv ? i - kKeys * 16 : i;
                const int key = e >> 4, cc = e & 15;
                const int64_t row = rr[key];
                const char* src = isv ? vb + row * v_row_stride * 2 + cc * 16 : kb + row * kv_row_stride * 2 + cc * 16;
                cp_async16(dst0 + (isv ? 2 * kBlock : 0) + (cc >> 3) * kBlock + key * 128 + (((cc & 7) ^ (key & 7)) << 4),
                           src);
            }
            cp_async_mbar_arrive_noinc(&c.xfull[stage]);
        }
        cp_async_wait_all();
        if (kPair) {
            cluster_wait();
            cluster_sync();
        }
    } else if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------------ MMA issuer
            const uint32_t idesc_qk = idesc_f16_f32_major(kKeys, kN, std::is_same<T, __nv_bfloat16>::value ? 1 : 0, 0, 0);
            const uint32_t idesc_pv = idesc_f16_f32_major(kD, kN, std::is_same<T, __nv_bfloat16>::value ? 1 : 0, 1, 0);
            const uint32_t qb = smem_u32(qs);
            bool ok = true;
            auto issue_qk = [&](int t) -> bool {
                const int stage = t % kStages;
                if (!mbar_wait(&c.xfull[stage], (uint32_t)((t / kStages) & 1))) return false;
                if (t >= 2 && !mbar_wait(&c.sempty[t & 1], (uint32_t)(((t - 2) >> 1) & 1))) return false;
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t kt = smem_u32(smem + (size_t)stage * kTile);
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint64_t ad = desc_sw128_kmajor(kt + (ks >> 2) * kBlock + (ks & 3) * 32, 1024);
                    const uint64_t bd = desc_sw128_kmajor(qb + (ks >> 2) * (kN * 128) + (ks & 3) * 32, 1024);
                    mma_f16_ss(tmem + (t & 1) * kN, ad, bd, idesc_qk, ks > 0 ? 1u : 0u);
                }
                mma_commit(&c.sfull[t & 1]);
                return true;
            };
            if (n_tiles > 0) ok = issue_qk(0);
            for (int t = 0; ok && t < n_tiles; ++t) {
                if (*(volatile int*)&c.abort) break;
                if (t + 1 < n_tiles && !issue_qk(t + 1)) {
                    ok = false;
                    break;
                }
                const int j = t & 1, stage = t % kStages;
                if (!mbar_wait(&c.pready[j], (uint32_t)((t >> 1) & 1))) {
                    ok = false;
                    break;
                }
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t vt = smem_u32(smem + (size_t)stage * kTile + 2 * kBlock);
                const uint32_t pb = smem_u32(ps + j * kPBytes);
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks) {
                    const uint64_t ad = desc_sw128_mnmajor(vt + ks * 2048, kBlock, 1024);
                    const uint64_t bd = desc_sw128_kmajor(pb + (ks >> 2) * (kN * 128) + (ks & 3) * 32, 1024);
                    mma_f16_ss(tmem + kOCol, ad, bd, idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(&c.xempty[stage]);
                mma_commit(&c.pvdone[j]);
            }
            if (!ok) abort_cta(c, g.status);
            mma_commit(&c.done);
            mbar_wait(&c.done, 0);
        }
        __syncwarp();
        if (kPair) {
            cluster_wait();
            cluster_sync();
        }
    } else {
        // ------------------------------------------------------------------ softmax (thread = key)
        const int quad = warp & 3;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int kk = quad * 32 + lane;          // this thread's key of a tile, and later its dim
        float m_used[kN], l_part[kN];
#pragma unroll
        for (int h = 0; h < kN; ++h) {
            m_used[h] = 0.f;
            l_part[h] = 0.f;
        }
        bool has_m = false, ok = true;
        uint32_t n_exch = 0;
        for (int t = 0; t < n_tiles; ++t) {
            const int j = t & 1;
            const uint32_t ph = (uint32_t)((t >> 1) & 1);
            if (warp_aborted(c) || !warp_wait(&c.sfull[j], ph)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float sv[kN];
            tmem_ld_32x32b_x16(tmem + lane_off + j * kN, sv);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.sempty[j]);
            const uint4 vm = *reinterpret_cast<const uint4*>(vmask + t * 4);
            const uint32_t vq = quad == 0 ? vm.x : quad == 1 ? vm.y : quad == 2 ? vm.z : vm.w;
            const bool valid = (vq >> lane) & 1u;
            const bool any_valid = (vm.x | vm.y | vm.z | vm.w) != 0u;
            // The running maximum of a head moves only when a key of the tile exceeds it by more than the
            // rescale margin.  Each warp first says whether one of its keys does (one vote); the maxima of
            // the tile are exchanged only then, and for the first tile with a valid key.
            bool over = false;
#pragma unroll
            for (int h = 0; h < kN; ++h) {
                sv[h] *= scale_log2;
                if (h < G && valid && sv[h] > m_used[h] + kRescaleLog2) over = true;
            }
            const bool w_over = __any_sync(0xffffffffu, over);
            if (lane == 0) c.over[j][quad] = w_over ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.rfull[j]);
            if (!warp_wait(&c.rfull[j], ph)) {
                ok = false;
                break;
            }
            const bool exch = any_valid && (!has_m || *reinterpret_cast<volatile uint32_t*>(c.over[j]) != 0u);
            if (exch) {
                // the tile's maximum per head over its 128 keys: warp maxima, exchanged through shared memory
#pragma unroll
                for (int h = 0; h < kN; ++h) {
                    if (h >= G) continue;   // (uniform)
                    float x = valid ? sv[h] : -3.0e38f;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
                    if (lane == 0) c.red[j][quad][h] = x;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.mfull);
                if (!warp_wait(&c.mfull, n_exch & 1u)) {
                    ok = false;
                    break;
                }
                ++n_exch;
            }
            float alpha[kN];
            bool resc = false;
#pragma unroll
            for (int h = 0; h < kN; ++h) {
                alpha[h] = 1.f;
                if (h >= G || !exch) continue;
                const float tmax = fmaxf(fmaxf(c.red[j][0][h], c.red[j][1][h]), fmaxf(c.red[j][2][h], c.red[j][3][h]));
                if (!has_m) {
                    m_used[h] = tmax;
                } else if (tmax > m_used[h] + kRescaleLog2) {
                    alpha[h] = ex2_approx(m_used[h] - tmax);
                    l_part[h] *= alpha[h];
                    m_used[h] = tmax;
                    resc = true;
                }
            }
            if (any_valid) has_m = true;
            if (resc && t > 0) {
                // this warp's lanes of O^T (thread = dim) once the PV MMAs of tile t-1 have completed
                const int tp = t - 1;
                if (!warp_wait(&c.pvdone[tp & 1], (uint32_t)((tp >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float o[kN];
                tmem_ld_32x32b_x16(tmem + lane_off + kOCol, o);
                tmem_ld_wait();
                uint32_t w[kN];
#pragma unroll
                for (int h = 0; h < kN; ++h) w[h] = __float_as_uint(o[h] * alpha[h]);
                tmem_st_32x32b_x16(tmem + lane_off + kOCol, w);
                tmem_st_wait();
            }
            // P^T tile j is free once the PV MMAs of tile t-2 have completed
            if (t >= 2 && !warp_wait(&c.pvdone[j], (uint32_t)(((t - 2) >> 1) & 1))) {
                ok = false;
                break;
            }
            uint8_t* pt = ps + j * kPBytes + (kk >> 6) * (kN * 128) + (kk & 7) * 2;
            const int chunk = (kk & 63) >> 3;
#pragma unroll
            for (int h = 0; h < kN; ++h) {
                if (h >= G) continue;
                const float p = (valid && has_m) ? ex2_approx(sv[h] - m_used[h]) : 0.f;
                l_part[h] += p;
                st_shared_u16(pt + h * 128 + ((chunk ^ (h & 7)) << 4), to_bits<T>(p));
            }
            fence_proxy_async_smem();   // P^T (generic stores) before the MMAs read it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.pready[j]);
        }
        if (!ok) abort_cta(c, g.status);
        // ------------------------------------------------------------------ output (thread = dim)
        // each head's row sum over the 128 key lanes
#pragma unroll
        for (int h = 0; h < kN; ++h) {
            if (h >= G) continue;
            float x = l_part[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (lane == 0) c.lred[quad][h] = x;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.lfull);
        bool have = ok && n_tiles > 0 && warp_wait(&c.lfull, 0);
        if (have) {
            const int tl = n_tiles - 1;
            have = warp_wait(&c.pvdone[tl & 1], (uint32_t)((tl >> 1) & 1));
            if (!have) abort_cta(c, g.status);
        }
        float o[kN];
#pragma unroll
        for (int h = 0; h < kN; ++h) o[h] = 0.f;
        if (have && !warp_aborted(c)) {
            tc_fence_after();
            tmem_ld_32x32b_x16(tmem + lane_off + kOCol, o);
            tmem_ld_wait();
        } else {
            have = false;
        }
        if (kPair) {
            cluster_wait();   // (phase 0: both CTAs have started)
            if (split == 1) {
#pragma unroll
                for (int h = 0; h < kN; ++h) {
                    if (h >= G) continue;
                    const float l = have ? (c.lred[0][h] + c.lred[1][h]) + (c.lred[2][h] + c.lred[3][h]) : 0.f;
                    st_cluster_f32(mapa(&c.xo[h][kk], 0), o[h]);
                    if (kk == 0) {
                        st_cluster_f32(mapa(&c.xml[h][0], 0), m_used[h] * 0.6931471805599453f);
                        st_cluster_f32(mapa(&c.xml[h][1], 0), l);
                    }
                }
            }
            cluster_sync();   // (phase 1: rank 1's output is in rank 0's shared memory)
            if (split == 0) {
#pragma unroll
                for (int h = 0; h < kN; ++h) {
                    if (h >= G) continue;
                    const float l0 = have ? (c.lred[0][h] + c.lred[1][h]) + (c.lred[2][h] + c.lred[3][h]) : 0.f;
                    const float m0 = m_used[h] * 0.6931471805599453f;
                    const float m1 = c.xml[h][0], l1 = c.xml[h][1];
                    float M = 0.f;
                    bool any = false;
                    if (l0 > 0.f) {
                        M = m0;
                        any = true;
                    }
                    if (l1 > 0.f) M = any ? fmaxf(M, m1) : m1;
                    float den = 0.f, acc = 0.f;
                    if (l0 > 0.f) den += expf(m0 - M) * l0;
                    if (l1 > 0.f) den += expf(m1 - M) * l1;
                    const float inv = den > 0.f ? 1.f / den : 0.f;
                    if (l0 > 0.f) acc += expf(m0 - M) * o[h];
                    if (l1 > 0.f) acc += expf(m1 - M) * c.xo[h][kk];
                    const int64_t dst = (r * Hq + h0 + h) * (int64_t)kD + kk;
                    if (out_dtype == IDX_BF16)
                        static_cast<__nv_bfloat16*>(out)[dst] = __float2bfloat16_rn(acc * inv);
                    else
                        static_cast<float*>(out)[dst] = acc * inv;
                }
            }
        }
#pragma unroll
        for (int h = 0; h < kN; ++h) {
            if (h >= G || kPair) continue;
            const float l = have ? (c.lred[0][h] + c.lred[1][h]) + (c.lred[2][h] + c.lred[3][h]) : 0.f;
            if (splits == 1) {
                const float val = l > 0.f ? o[h] / l : 0.f;
                const int64_t dst = (r * Hq + h0 + h) * (int64_t)kD + kk;
                if (out_dtype == IDX_BF16)
                    static_cast<__nv_bfloat16*>(out)[dst] = __float2bfloat16_rn(val);
                else
                    static_cast<float*>(out)[dst] = val;
            } else {
                // the split's unnormalised output, maximum (natural-log units) and sum
                const int64_t u = (r * splits + split) * (int64_t)Hq + h0 + h;
                part_o[u * kD + kk] = o[h];
                if (kk == 0) {
                    part_ml[2 * u] = m_used[h] * 0.6931471805599453f;
                    part_ml[2 * u + 1] = l;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool gqa_tc_supported(int dtype, int Hq, int Hkv, int dk, int dv, const void* k, const void* v,
                      int64_t kv_row_stride, int64_t v_row_stride, const void* q) {
    return (dtype == IDX_BF16 || dtype == IDX_F16) && v && dk == kD && dv == kD && Hkv >= 1 && Hq % Hkv == 0 &&
           Hq / Hkv <= kN && kv_row_stride % 8 == 0 && v_row_stride % 8 == 0 &&
           !(reinterpret_cast<uintptr_t>(k) & 15u) && !(reinterpret_cast<uintptr_t>(v) & 15u) &&
           !(reinterpret_cast<uintptr_t>(q) & 15u);
}

// key splits per (row, kv head): one CTA per SM when the (row, kv head) units are few, at least 256
// selected keys and at most kMaxKps per split
int gqa_tc_splits(int64_t units, int64_t cap) {
    const int64_t min_s = (cap + kMaxKps - 1) / kMaxKps;
    int sms = sm_count();
    if (sms < 2) sms = 152;
    int64_t s = units > 0 ? sms / units : 1;
    const int64_t by_keys = (cap + 255) / 256;
    if (s > by_keys) s = by_keys;
    if (s < min_s) s = min_s;
    return s < 1 ? 1 : (int)s;
}

namespace {

// the kernel with programmatic stream serialisation, as 2-CTA clusters when kPair
template <typename T, bool kPair>
cudaError_t launch_gqa(int64_t grid, const void* q, const void* k, const void* v, int64_t kv_row_stride,
                       int64_t v_row_stride, int64_t kv_rows, const Geom& g, const int32_t* idx, int64_t idx_row_stride,
                       const int32_t* n_sel, int Hq, int Hkv, float scale_log2, int splits, int kps, void* out,
                       int out_dtype, float* part_o, float* part_ml, cudaStream_t st) {
    auto kern = attn_gqa_tc_kernel<T, kPair>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kPair ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kPair ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const T*>(q), static_cast<const T*>(k),
                              static_cast<const T*>(v), kv_row_stride, v_row_stride, kv_rows, g, idx, idx_row_stride,
                              n_sel, Hq, Hkv, scale_log2, splits, kps, out, out_dtype, part_o, part_ml);
}

}  // namespace

cudaError_t launch_attn_gqa_tc(const void* q, int dtype, int Hq, int Hkv, const void* k, const void* v,
                               int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                               const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel, float scale,
                               void* out, int out_dtype, void* ws, size_t ws_bytes, cudaStream_t st) {
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0) return cudaSuccess;
    if (kv_rows < 1 || kv_rows > INT32_MAX) return cudaErrorNotSupported;   // (padding gathers row 0 or later)
    int splits = gqa_tc_splits(n_rows * Hkv, idx_row_stride);
    const size_t per_split = (size_t)n_rows * Hq * (kD + 2) * sizeof(float);
    const int64_t min_s = (idx_row_stride + kMaxKps - 1) / kMaxKps;
    if (splits > 1) {
        const int64_t fit = (ws && !(reinterpret_cast<uintptr_t>(ws) & 15u)) ? (int64_t)(ws_bytes / per_split) : 0;
        if (fit < splits) splits = (int)(fit > 1 ? fit : 1);
    }
    if (splits < min_s) return cudaErrorNotSupported;   // (the CUDA-core path takes it)
    const int kps = (int)(((idx_row_stride + splits - 1) / splits + kKeys - 1) / kKeys * kKeys);
    if (kps > kMaxKps) return cudaErrorNotSupported;
    const int64_t grid = n_rows * Hkv * splits;
    if (grid > INT32_MAX) return cudaErrorNotSupported;
    // two splits: a 2-CTA cluster per (row, kv head) merges them itself; more: partials + combine
    const bool pair = splits == 2;
    float* part_o = splits > 2 ? static_cast<float*>(ws) : nullptr;
    float* part_ml = splits > 2 ? part_o + (size_t)n_rows * splits * Hq * kD : nullptr;
    const float scale_log2 = scale * 1.4426950408889634f;
    cudaError_t e;
    if (dtype == IDX_BF16)
        e = pair ? launch_gqa<__nv_bfloat16, true>(grid, q, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                                                   idx_row_stride, n_sel, Hq, Hkv, scale_log2, splits, kps, out,
                                                   out_dtype, part_o, part_ml, st)
                 : launch_gqa<__nv_bfloat16, false>(grid, q, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                                                    idx_row_stride, n_sel, Hq, Hkv, scale_log2, splits, kps, out,
                                                    out_dtype, part_o, part_ml, st);
    else
        e = pair ? launch_gqa<__half, true>(grid, q, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                                            idx_row_stride, n_sel, Hq, Hkv, scale_log2, splits, kps, out, out_dtype,
                                            part_o, part_ml, st)
                 : launch_gqa<__half, false>(grid, q, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                                             idx_row_stride, n_sel, Hq, Hkv, scale_log2, splits, kps, out, out_dtype,
                                             part_o, part_ml, st);
    if (e != cudaSuccess || splits <= 2) return e;
    return launch_attn_generic_combine(part_o, part_ml, splits, n_rows, Hq, kD, out, out_dtype, st);
}

}  // namespace lidx
