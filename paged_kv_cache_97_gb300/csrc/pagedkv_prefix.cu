// pagedkv_prefix.cu -- attention of every sequence's query rows over a
// shared prefix of physical blocks.
//
// When the first P blocks of every sequence's block table are the same
// physical blocks (a shared system prompt: “让 Agent 跑得快”, §五 共享前缀 --
// several block tables map to the same read-only blocks), the prefix part of
// attention is one dense product per KV head h:
//   S[rows x tokens] = Q_h[rows x d] . K_prefix^T,   O = softmax-weighted V
// with rows = (sequence, grouped query head) over the whole batch.  This
// kernel computes it once per head instead of once per sequence: the prefix
// K/V is read from HBM once and every CTA re-reads only its 16-token blocks
// through L2.  The online-softmax partial (m, l, unnormalised acc) of each
// row and prefix chunk goes to the row's partial slots; the decode kernel
// covers tokens past the prefix and the merge kernel combines both
// (“LLM 推理优化技术全景”, 在线 Softmax; “Flash Attention v2 的改进”).
//
// Tiling: a CTA of 4 warps takes 64 rows (16 per warp, the M of
// mma.sync m16n8k16) of one KV head and one chunk of the prefix blocks; the
// blocks stream through a 4-stage ring of TMA tensor loads.  Per 16-token
// tile a warp computes S = Q . K^T (two n-tiles of 8 tokens), updates the
// online softmax per row, and reuses the S accumulator registers as the A
// operand of O += P . V (the fragment layouts coincide), V^T fragments coming
// from ldmatrix.trans.  bf16 pools only.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {
namespace {

using namespace dev;

constexpr int kPWarps = 4;
constexpr int kPThreads = kPWarps * 32;
constexpr int kPRows = kPWarps * 16;     // query rows per CTA
constexpr int kPStages = 4;

template <int D, int BS>
__global__ void __launch_bounds__(kPThreads)
    prefix_kernel(const __grid_constant__ CUtensorMap k_map,
                  const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  using G = Geo<D, BS, false>;
  constexpr int S = kPStages;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S];
  __shared__ int cta_bad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads, GQ = Hq / Hkv;
  const int hk = blockIdx.y, chunk = blockIdx.z;
  const int rows_total = a.batch * GQ;
  const int P = a.num_prefix_blocks, nc = a.prefix_chunks;
  const int c0 = (int)((int64_t)chunk * P / nc), c1 = (int)((int64_t)(chunk + 1) * P / nc);
  const int n = c1 - c0;                                  // >= 1 (nc <= P)
  const uint32_t stages = (smem_addr(smem_raw) + 1023u) & ~1023u;
  // The decode kernel queued behind this one needs nothing from it: let it
  // start now (the merge, a plain launch, waits for both).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (tid == 0) {
    cta_bad = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kPWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // This warp's rows ra = r0 + g and rb = r0 + g + 8: (sequence, query head).
  const int r0 = blockIdx.x * kPRows + warp * 16;
  const int ra = r0 + g, rb = ra + 8;
  const bool va = ra < rows_total, vb = rb < rows_total;
  const int64_t qrow_a = va ? ((int64_t)(ra / GQ) * Hq + (int64_t)hk * GQ + ra % GQ) : 0;
  const int64_t qrow_b = vb ? ((int64_t)(rb / GQ) * Hq + (int64_t)hk * GQ + rb % GQ) : 0;
  // Q A-fragments: a0 = (row g, d 16ks+2t..+1), a1 = (row g+8, same d),
  // a2 = (row g, d 16ks+2t+8..+9), a3 = (row g+8, same d).
  uint32_t qa[G::kKSteps][4];
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
    for (int ks = 0; ks < G::kKSteps; ++ks) {
      const int d0 = 16 * ks + 2 * t;
      qa[ks][0] = va ? *reinterpret_cast<const uint32_t*>(q + qrow_a * D + d0) : 0u;
      qa[ks][1] = vb ? *reinterpret_cast<const uint32_t*>(q + qrow_b * D + d0) : 0u;
      qa[ks][2] = va ? *reinterpret_cast<const uint32_t*>(q + qrow_a * D + d0 + 8) : 0u;
      qa[ks][3] = vb ? *reinterpret_cast<const uint32_t*>(q + qrow_b * D + d0 + 8) : 0u;
    }
  }
  __syncthreads();                                        // barriers initialised
  for (int j = c0 + tid; j < c1; j += kPThreads) {
    const int32_t p = a.prefix_blocks[j];
    if (p < 0 || p >= a.num_blocks) cta_bad = 1;
  }
  __syncthreads();
  const bool bad = cta_bad != 0;

  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  bool ok = true;

  auto issue = [&](int k) {                               // thread 0 only
    const int s = k % S;
    if (k >= S && !mbar_wait(smem_addr(&empty_bar[s]), ((k / S) - 1) & 1)) return false;
    const int p = a.prefix_blocks[c0 + k];
    const uint32_t fb = smem_addr(&full_bar[s]);
    mbar_expect_tx(fb, (uint32_t)G::kBlockBytes);
    const uint32_t kdst = stages + (uint32_t)(s * G::kBlockBytes);
    const uint32_t vdst = kdst + G::kTensorBytes;
#pragma unroll
    for (int x = 0; x < G::kBoxes; ++x) {
      tma_load_4d(kdst + x * G::kBoxBytes, &k_map, fb, x * G::kBoxElems, hk, 0, p);
      tma_load_4d(vdst + x * G::kBoxBytes, &v_map, fb, x * G::kBoxElems, hk, 0, p);
    }
    return true;
  };

  int issued = 0;
  if (!bad) {
    if (tid == 0)
      for (int k = 0; k < S - 1 && k < n; ++k) ok = ok && issue(k);
    issued = min(S - 1, n);
    for (int k = 0; k < n; ++k) {
      if (tid == 0 && k + S - 1 < n) ok = ok && issue(k + S - 1);
      issued = min(n, k + S);
      const int s = k % S;
      if (!mbar_wait(smem_addr(&full_bar[s]), (k / S) & 1)) {
        ok = false;
        break;
      }
      const uint32_t kb = stages + (uint32_t)(s * G::kBlockBytes), vb = kb + G::kTensorBytes;
#pragma unroll
      for (int tile = 0; tile < G::kTiles; ++tile) {
        // ---- S = Q . K^T for 16 tokens: n-tiles of tokens 0-7 and 8-15.
        // ldmatrix.x4 matrix q = lane/8: tokens 8*(q>>1)..+7, d-chunk
        // 2ks + (q&1) -> b0, b1 of n-tile 0, then of n-tile 1.
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = tile * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < G::kKSteps; ++ks) {
          uint32_t fb4[4];
          ldsm_x4(fb4, kb + chunk_off<G>(krow, 2 * ks + ((lane >> 3) & 1)));
          mma16816<false>(c[0], qa[ks], fb4[0], fb4[1]);
          mma16816<false>(c[1], qa[ks], fb4[2], fb4[3]);
        }
        // ---- online softmax per row (rows g: c[.][0..1], g+8: c[.][2..3])
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) c[nt][e] *= a.scale_log2;
        float mx_a = fmaxf(fmaxf(c[0][0], c[0][1]), fmaxf(c[1][0], c[1][1]));
        float mx_b = fmaxf(fmaxf(c[0][2], c[0][3]), fmaxf(c[1][2], c[1][3]));
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
          mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
          mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
        }
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float al_a = exp2f(m_a - mn_a), al_b = exp2f(m_b - mn_b);
        m_a = mn_a;
        m_b = mn_b;
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          p[nt][0] = exp2f(c[nt][0] - mn_a);
          p[nt][1] = exp2f(c[nt][1] - mn_a);
          p[nt][2] = exp2f(c[nt][2] - mn_b);
          p[nt][3] = exp2f(c[nt][3] - mn_b);
        }
        l_a = l_a * al_a + p[0][0] + p[0][1] + p[1][0] + p[1][1];
        l_b = l_b * al_b + p[0][2] + p[0][3] + p[1][2] + p[1][3];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
          o[i][0] *= al_a;
          o[i][1] *= al_a;
          o[i][2] *= al_b;
          o[i][3] *= al_b;
        }
        // ---- O += P . V: P's A fragment is the S accumulator layout.
        const uint32_t pa[4] = {pack2<false>(p[0][0], p[0][1]), pack2<false>(p[0][2], p[0][3]),
                                pack2<false>(p[1][0], p[1][1]), pack2<false>(p[1][2], p[1][3])};
        // ldmatrix.x4.trans matrix q = lane/8: tokens 8*(q&1)..+7, d-chunk
        // 2jj + (q>>1) -> b0, b1 of d n-tile 2jj, then of 2jj+1.
        const int vrow = tile * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t fb4[4];
          ldsm_x4_t(fb4, vb + chunk_off<G>(vrow, 2 * jj + (lane >> 4)));
          mma16816<false>(o[2 * jj], pa, fb4[0], fb4[1]);
          mma16816<false>(o[2 * jj + 1], pa, fb4[2], fb4[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
    }
    if (tid == 0) {
      // Let every issued fill land before the CTA may exit (bounded): wait
      // for the last fill of each stage (earlier phases are complete).
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = s + S * ((issued - 1 - s) / S);
        if (!mbar_wait(smem_addr(&full_bar[s]), (last / S) & 1)) ok = false;
      }
    }
  }
  if (!ok) atomicOr(a.flags, PAGEDKV_FLAG_WAIT_TIMEOUT);
  if (bad && tid == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_BLOCK);

  // ---- the rows' partials for this chunk (slot max_parts + chunk)
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  const bool failed = bad || !ok;
  const int slot = a.max_parts + chunk;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const bool v = half ? vb : va;
    if (!v) continue;
    const int64_t r = (half ? qrow_b : qrow_a) * a.slots + slot;
    if (t == 0) {
      a.ws_ml[2 * r] = half ? m_b : m_a;
      a.ws_ml[2 * r + 1] = failed ? -1.0f : (half ? l_b : l_a);
    }
    float* acc = a.ws_acc + r * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<float2*>(acc + 8 * i + 2 * t) =
          make_float2(o[i][2 * half], o[i][2 * half + 1]);
  }
}

template <int D, int BS>
kv_status launch_p(const DecodeArgs& a, cudaStream_t s) {
  using G = Geo<D, BS, false>;
  constexpr int kSmem = kPStages * G::kBlockBytes + 1024;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      st = cuda_check(cudaFuncSetAttribute(prefix_kernel<D, BS>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem),
                      "cudaFuncSetAttribute(prefix_kernel)");
      if (st != KV_OK) return st;
      attr_set[dev] = true;
    }
  }
  alignas(64) CUtensorMap km, vm;
  if ((st = make_kv_maps(a, &km, &vm)) != KV_OK) return st;
  const int GQ = a.num_q_heads / a.num_kv_heads;
  const dim3 grid((unsigned)((a.batch * GQ + kPRows - 1) / kPRows), (unsigned)a.num_kv_heads,
                  (unsigned)a.prefix_chunks);
  prefix_kernel<D, BS><<<grid, kPThreads, kSmem, s>>>(km, vm, a);
  return cuda_check(cudaGetLastError(), "prefix_kernel launch");
}

}  // namespace

kv_status launch_prefix(const DecodeArgs& a, cudaStream_t s) {
  if (a.dtype != KV_DTYPE_BF16)
    return fail(KV_ERR_NOT_IMPLEMENTED, "the shared-prefix path supports bf16 pools only");
  if (a.prefix_chunks < 1 || a.prefix_chunks > a.num_prefix_blocks)
    return fail(KV_ERR_INVALID_ARG, "bad prefix chunk count");
  if (a.head_dim == 128) return a.block_size == 32 ? launch_p<128, 32>(a, s) : launch_p<128, 16>(a, s);
  return a.block_size == 32 ? launch_p<64, 32>(a, s) : launch_p<64, 16>(a, s);
}

}  // namespace pagedkv
