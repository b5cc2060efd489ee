// The sparse MLA attention kernel (one work unit per 2-CTA cluster) and the
// merge of key splits; the unit's device code is in attn_mla_tc.cuh.
#include "attn_mla_tc.cuh"

namespace lidx {
namespace {
using namespace sm100;

// A persistent grid of 2-CTA clusters: cluster c runs the units c, c + C, c + 2C, ... (C clusters),
// keeping its TMEM and re-initialising its barriers between units (every phase of the last unit has
// completed and no remote arrival is pending once both CTAs passed the unit's closing cluster barrier).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_attn_tc_kernel(const __nv_bfloat16* __restrict__ lat, int64_t lat_row_stride,
                       const __nv_bfloat16* __restrict__ q, Geom g, const int32_t* idx,
                       int64_t idx_row_stride, const int32_t* n_sel, int64_t kv_rows,
                       float scale_log2, int splits, int kps, void* __restrict__ out, int out_dtype,
                       float* __restrict__ part_o, float* __restrict__ part_ml, int64_t n_units) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const MlaSmem sm = mla_smem(smem);
    Ctl& c = *sm.c;
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5;
    const int64_t n_clusters = gridDim.x >> 1;
    pdl_trigger();

    if (threadIdx.x == 0) mla_init(c);
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;

    const bool q_warp = mla_q_warp(rank);
    for (int64_t unit = blockIdx.x >> 1; unit < n_units; unit += n_clusters) {
        const bool first = unit == (int64_t)(blockIdx.x >> 1);
        if (!first) {
            if (threadIdx.x == 0) mla_init(c);
            __syncthreads();
        }
        // Rank 0's softmax warps put Q into TMEM (Q is an input no other kernel writes, so for the
        // first unit this overlaps the end of the previous kernel) while the other warps, once the
        // previous kernel's selection is visible, stage the split's selected keys.
        if (q_warp) mla_load_q(c, sm.xtiles, tmem, q, unit / splits);
        if (first) pdl_wait();
        const Unit u = make_unit(unit, g, n_sel, idx_row_stride, kv_rows, splits, kps);
        if (!q_warp) mla_stage_rows(sm, rank, u, g, idx, idx_row_stride, kv_rows);
        tc_fence_before();
        cluster_sync();  // barriers of both CTAs initialised, indices staged
        tc_fence_after();
        mla_run(sm, tmem, rank, u, unit, lat, lat_row_stride, g, scale_log2, splits, out, out_dtype, part_o, part_ml);
        tc_fence_before();
        __syncthreads();
        cluster_sync();  // no cross-CTA traffic of this unit is in flight
        tc_fence_after();
    }
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Merge key splits: out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s over splits with l_s > 0.
__global__ void __launch_bounds__(128) mla_combine_kernel(const float* part_o,
                                                          const float* part_ml, int splits,
                                                          void* __restrict__ out, int out_dtype) {
    pdl_trigger();
    pdl_wait();
    // block (row, 4 columns), thread = head: the partials ([unit][column / 4][head][4]) are read
    // coalesced, 16 bytes per head and split
    const int64_t r = blockIdx.x;
    const int c0 = blockIdx.y * 4;
    const int h = threadIdx.x;
    float M = -3.0e38f;
    bool any = false;
    for (int s = 0; s < splits; ++s) {
        const int64_t u = r * splits + s;
        const float l = part_ml[(u * kHq + h) * 2 + 1];
        if (l > 0.f) {
            M = fmaxf(M, part_ml[(u * kHq + h) * 2]);
            any = true;
        }
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float den = 0.f;
    if (any) {
        for (int s = 0; s < splits; ++s) {
            const int64_t u = r * splits + s;
            const float l = part_ml[(u * kHq + h) * 2 + 1];
            if (!(l > 0.f)) continue;
            const float wgt = exp2f(part_ml[(u * kHq + h) * 2] - M);
            den += wgt * l;
            const float4 o = reinterpret_cast<const float4*>(part_o + u * (int64_t)kDv * kHq)[(c0 / 4) * kHq + h];
            acc[0] += wgt * o.x;
            acc[1] += wgt * o.y;
            acc[2] += wgt * o.z;
            acc[3] += wgt * o.w;
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int64_t base = (r * kHq + h) * (int64_t)kDv + c0;
    if (out_dtype == IDX_BF16) {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + base;
        *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
        *reinterpret_cast<__nv_bfloat162*>(o + 2) = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + base) =
            make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    }
}

}  // namespace

// key splits per query row: enough clusters to cover the SMs when rows are few,
// and never more than kMaxKps selected keys per split
int mla_splits(int64_t n_rows, int64_t cap) {
    const int64_t min_s = cap > kMaxKps ? (cap + kMaxKps - 1) / kMaxKps : 1;
    if (n_rows <= 0) return (int)min_s;
    int sms = sm_count();
    if (sms < 2) sms = 152;
    const int64_t clusters = sms / 2;
    int64_t s = 1;
    if (n_rows < clusters) {
        const int64_t by_sm = clusters / n_rows;
        const int64_t by_keys = (cap + 255) / 256;
        s = by_sm < by_keys ? by_sm : by_keys;
    }
    if (s < min_s) s = min_s;
    return (int)(s < 1 ? 1 : s);
}

size_t mla_workspace_bytes(int64_t n_rows, int64_t cap) {
    const int s = mla_splits(n_rows, cap);
    if (s <= 1) return 0;
    return (size_t)n_rows * s * kHq * (kDv + 2) * sizeof(float);
}

// clusters of the attention kernel that can be resident at once (0: unknown)
int64_t mla_clusters() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev]) return cache[dev] > 0 ? cache[dev] : 0;
    cudaFuncSetAttribute(mla_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mla_attn_tc_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[dev] = n > 0 ? n : -1;
    return n > 0 ? n : 0;
}

bool mla_tc_supported(int dtype, int Hq, int Hkv, int dk, int dv, const void* k, const void* v,
                      int64_t kv_row_stride, int64_t kv_rows, const void* q, const void* out) {
    return dtype == IDX_BF16 && !v && Hq == kHq && Hkv == 1 && dk == kDk && dv == kDv &&
           kv_row_stride % 8 == 0 && kv_rows >= 1 && kv_rows <= INT32_MAX &&
           !(reinterpret_cast<uintptr_t>(k) & 15u) && !(reinterpret_cast<uintptr_t>(q) & 15u) &&
           !(reinterpret_cast<uintptr_t>(out) & 15u);
}

cudaError_t launch_attn_mla_tc(const void* q, const void* lat, int64_t kv_row_stride, int64_t kv_rows,
                               const Geom& g, const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel,
                               float scale, void* out, int out_dtype, void* ws, size_t ws_bytes,
                               cudaStream_t st) {
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0) return cudaSuccess;
    const int splits = mla_splits(n_rows, idx_row_stride);
    const int64_t kps64 = ((idx_row_stride + splits - 1) / splits + kKeys - 1) / kKeys * kKeys;
    float* part_o = nullptr;
    float* part_ml = nullptr;
    if (splits > 1) {
        const size_t need = mla_workspace_bytes(n_rows, idx_row_stride);
        if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u)) return cudaErrorInvalidValue;
        part_o = static_cast<float*>(ws);
        part_ml = part_o + (size_t)n_rows * splits * kHq * kDv;
    }
    const int64_t n_units = n_rows * splits;
    cudaFuncSetAttribute(mla_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    const int64_t resident = mla_clusters();
    const int64_t clusters = resident > 0 && resident < n_units ? resident : n_units;
    const float scale_log2 = scale * 1.4426950408889634f;
    cudaError_t e = launch_pdl(mla_attn_tc_kernel, dim3((unsigned)(2 * clusters)), dim3(kThreads), kSmemBytes, st,
                               static_cast<const __nv_bfloat16*>(lat), kv_row_stride,
                               static_cast<const __nv_bfloat16*>(q), g, idx, idx_row_stride, n_sel, kv_rows,
                               scale_log2, splits, (int)kps64, out, out_dtype, part_o, part_ml, n_units);
    if (e != cudaSuccess || splits == 1) return e;
    return launch_pdl(mla_combine_kernel, dim3((unsigned)n_rows, kDv / 4), dim3(kHq), 0, st,
                      static_cast<const float*>(part_o), static_cast<const float*>(part_ml), splits, out, out_dtype);
}

}  // namespace lidx
