// Template dispatch of the decode kernels over head_dim and padded group size.
#pragma once

#include "decode.cuh"
#include "decode_mma.cuh"
#include "decode_prefix.cuh"
#include "decode_sk.cuh"
#include "launch.h"

namespace pkv {

// Raises the dynamic shared-memory limit of a kernel once per device.
template <typename K>
cudaError_t configure_once(K kern, size_t smem, bool (&configured)[kMaxDevices]) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    configured[dev] = true;
  }
  return cudaSuccess;
}

// Shape of the one-CTA-per-(sequence, KV head, partition) kernels: warps per
// CTA and stages per warp. The CUDA-core kernel takes 4 warps x 2 stages.
// The tensor-core (group size >= 2) kernel takes 3 warps x 2 stages (48 KB of
// ring, 4 CTAs per SM). Measured on GB300, Llama-3-8B-shaped layer with the
// shortest sequences last and partial-tile boxes: 41.4 us with 4 x 2, 40.2-40.3
// with 3 x 2; three-stage rings (4 x 3, 3 x 3) and 2 x 4 were 46-52 us.
constexpr int kGridWarps = 4;
constexpr int kGridStages = 2;
constexpr int kMmaWarps = 3;
constexpr int kMmaStages = 2;
// The shared-prefix schedule's CTAs (group rows) take 2 warps x 2 stages:
// 32 KB of ring and 168 registers a thread hold 6 CTAs per SM (912), so the
// LLaMA-13B beam batch's 640 group CTAs run in one wave: 57.0 us against
// 59.5 us with 3 x 2 (4 per SM); the OPT-66B sampling batch (2304 group CTAs)
// is 233.0 us either way. The plan's split rule still counts slots of the
// 3 x 2 CTA (one wave of that shape's in-flight bytes): counting the 912 of
// this one split the beam batch's groups and took 61.3 us.
constexpr int kPrefixWarps = 2;
constexpr int kPrefixStages = 2;

// Launch with programmatic stream serialization: the grid may become resident
// while the previous kernel in the stream finishes (the kernels wait for it
// with griddepcontrol.wait before touching global memory).
template <typename K, typename... Args>
cudaError_t launch_pdl(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Ring shape of the CUDA-core kernel for wide grids: with at least
// kWideGridCtas CTAs (13+ waves; the OPT-66B parallel-sampling batch has
// 9216) six warps with one stage each -- 4 CTAs, 24 warps per SM instead of
// 3 CTAs of 4 warps x 2 stages -- hide latency better: measured on GB300,
// 341 -> 299 us on that batch, whose sibling samples share prompt blocks
// through L2, against 1-1.4 % slower on the LLaMA-13B and OPT-175B layers,
// which keep the two-stage ring.
constexpr int kWideGridWarps = 6;
constexpr int64_t kWideGridCtas = 8192;
// One-pass CUDA-core grids of at most kLongGridCtas CTAs (under two waves of
// 4 x 2 CTAs at 3 per SM) hold few, long CTAs, and the longest CTA's own rate
// (its share of its SM's copies: a third at 3 CTAs per SM) nears the whole
// call: there the CTAs take 6 warps x 2 stages (2 per SM, the same 12 warps
// and 192 KB of ring per SM). Measured on GB300, OPT-175B layer (768 CTAs):
// 1177.0-1177.5 us with 4 x 2, 1160.4-1160.8 with 6 x 2, 1177.5-1177.9 with
// 4 x 3 and 5 x 2, 1220.5-1221.0 with 3 x 2; LLaMA-13B layer (2560 CTAs):
// 132.2-132.4 us with 4 x 2 against 133.7-133.8 with 6 x 2.
// Split-K grids of at most kLongGridCtas CTAs take the same shape only when
// their partitions are long: the first N sequences of the OPT-175B layer, 768
// CTAs (672 for N = 1), 4 x 2 against 6 x 2: N = 4 (15168-token partitions)
// 726.1 -> 713.7 us, N = 2 (7584) 396.9 -> 409.7 us, N = 1 (4336) 222.7 ->
// 233.9 us; the change of sign lies near 12K tokens.
constexpr int kLongGridWarps = 6;
constexpr int64_t kLongGridCtas = 1024;
constexpr int kLongSplitTokens = 12288;

template <typename T, int D, int G, int NW, int STAGES>
cudaError_t launch_cuda_core_grid(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
  using C = DecodeCfg<T, D, G, NW, STAGES>;
  auto kern = paged_decode_kernel<T, D, G, NW, STAGES>;
  static bool configured[kMaxDevices] = {};
  cudaError_t err = configure_once(kern, C::SMEM_BYTES, configured);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, grid, dim3(NW * 32), C::SMEM_BYTES, stream, a);
}

template <typename T, int D, int G, int MW, int MS>
cudaError_t launch_mma_grid(const DecodeArgs& a, dim3 grid, const CUtensorMap* kmap, const CUtensorMap* vmap,
                            cudaStream_t stream) {
  using C = MmaCfg<T, D, MW, MS>;
  auto kern = paged_decode_mma_kernel<T, D, G, MW, MS>;
  static bool configured[kMaxDevices] = {};
  cudaError_t err = configure_once(kern, C::SMEM_BYTES, configured);
  if (err != cudaSuccess) return err;
  PoolMaps maps;
  for (int i = 0; i < 3; ++i) {
    maps.k[i] = kmap[i];
    maps.v[i] = vmap[i];
  }
  return launch_pdl(kern, grid, dim3(MW * 32), C::SMEM_BYTES, stream, a, maps);
}

template <typename T, int D, int G>
cudaError_t launch_decode_dg(const DecodeArgs& a, const CUtensorMap* kmap, const CUtensorMap* vmap,
                             cudaStream_t stream) {
  constexpr int NW = kGridWarps;
  constexpr int STAGES = kGridStages;
  // (the shared-prefix schedule: rows for its chunks, then the sequences, one pass)
  const dim3 grid(unsigned(a.num_kv_heads), unsigned(a.num_seqs + (a.prefix_header ? a.prefix_slots : 0)),
                  a.prefix_header ? 1u : unsigned(a.max_parts));
  if constexpr (G == 1) {
    const int64_t ctas = int64_t(grid.x) * grid.y * grid.z;
    const bool long_ctas = grid.z == 1 || a.part_tokens >= kLongSplitTokens;
    const bool long_grid = long_ctas && !a.prefix_header && ctas <= kLongGridCtas;
    cudaError_t err = ctas >= kWideGridCtas ? launch_cuda_core_grid<T, D, G, kWideGridWarps, 1>(a, grid, stream)
                      : long_grid           ? launch_cuda_core_grid<T, D, G, kLongGridWarps, STAGES>(a, grid, stream)
                                            : launch_cuda_core_grid<T, D, G, NW, STAGES>(a, grid, stream);
    if (err != cudaSuccess) return err;
  } else {
    cudaError_t err;
    if constexpr (G == kPrefixRows) {
      err = a.prefix_header ? launch_mma_grid<T, D, G, kPrefixWarps, kPrefixStages>(a, grid, kmap, vmap, stream)
                            : launch_mma_grid<T, D, G, kMmaWarps, kMmaStages>(a, grid, kmap, vmap, stream);
    } else {
      err = launch_mma_grid<T, D, G, kMmaWarps, kMmaStages>(a, grid, kmap, vmap, stream);
    }
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

// Slots the shared-prefix plan splits groups against: CTAs of the 3 x 2
// group-row kernel that one SM holds at once, times the SMs of the current
// device (the group CTAs themselves run 2 x 2, see kPrefixWarps).
template <typename T, int D>
cudaError_t prefix_resident_ctas_d(int* ctas) {
  using C = MmaCfg<T, D, kMmaWarps, kMmaStages>;
  auto kern = paged_decode_mma_kernel<T, D, kPrefixRows, kMmaWarps, kMmaStages>;
  static bool configured[kMaxDevices] = {};
  cudaError_t err = configure_once(kern, C::SMEM_BYTES, configured);
  if (err != cudaSuccess) return err;
  int per_sm = 0, dev = 0, sms = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMmaWarps * 32, C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  *ctas = per_sm * sms;
  return cudaSuccess;
}

template <typename T, int D>
cudaError_t launch_decode_d(const DecodeArgs& a, int gpad, const CUtensorMap* kmap, const CUtensorMap* vmap,
                            cudaStream_t stream) {
  switch (gpad) {
    case 1: return launch_decode_dg<T, D, 1>(a, kmap, vmap, stream);
    case 2: return launch_decode_dg<T, D, 2>(a, kmap, vmap, stream);
    case 4: return launch_decode_dg<T, D, 4>(a, kmap, vmap, stream);
    case 8: return launch_decode_dg<T, D, 8>(a, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_decode_t(const DecodeArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                            const CUtensorMap* vmap, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_decode_d<T, 64>(a, gpad, kmap, vmap, stream);
    case 128: return launch_decode_d<T, 128>(a, gpad, kmap, vmap, stream);
    case 256: return launch_decode_d<T, 256>(a, gpad, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ---- balanced persistent schedule -------------------------------------------
template <typename T, int D, int G>
cudaError_t launch_decode_sk_dg(const SkArgs& a, const CUtensorMap* kmap, const CUtensorMap* vmap,
                                cudaStream_t stream) {
  constexpr int NW = sk_warps<D, G>();
  constexpr int STAGES = sk_stages<D>();
  constexpr bool MMA = G > 1;
  using SM = SkSmem<T, D, G, NW, STAGES, MMA>;
  auto kern = paged_decode_sk_kernel<T, D, G, NW, STAGES, MMA>;
  static bool configured[kMaxDevices] = {};
  static int sm_count[kMaxDevices] = {};
  if (a.num_seqs > SM::max_seqs()) return cudaErrorInvalidValue;
  cudaError_t err = configure_once(kern, SM::bytes(SM::max_seqs()), configured);
  if (err != cudaSuccess) return err;
  int dev = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (!sm_count[dev]) {
    err = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
  }
  const size_t smem = SM::bytes(a.num_seqs);
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem);
  if (err != cudaSuccess) return err;
  int grid = sm_count[dev] * (per_sm > 0 ? per_sm : 1);
  if (grid > kSkMaxWarps / NW) grid = kSkMaxWarps / NW;
  err = launch_pdl(kern, dim3(grid), dim3(NW * 32), smem, stream, a, *kmap, *vmap);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <typename T, int D>
int sk_max_seqs_d(int gpad) {
  switch (gpad) {
    case 1: return SkSmem<T, D, 1, sk_warps<D, 1>(), sk_stages<D>(), false>::max_seqs();
    case 2: return SkSmem<T, D, 2, sk_warps<D, 2>(), sk_stages<D>(), true>::max_seqs();
    case 4: return SkSmem<T, D, 4, sk_warps<D, 4>(), sk_stages<D>(), true>::max_seqs();
    case 8: return SkSmem<T, D, 8, sk_warps<D, 8>(), sk_stages<D>(), true>::max_seqs();
    default: return 0;
  }
}

template <typename T, int D>
cudaError_t launch_decode_sk_d(const SkArgs& a, int gpad, const CUtensorMap* kmap, const CUtensorMap* vmap,
                               cudaStream_t stream) {
  switch (gpad) {
    case 1: return launch_decode_sk_dg<T, D, 1>(a, kmap, vmap, stream);
    case 2: return launch_decode_sk_dg<T, D, 2>(a, kmap, vmap, stream);
    case 4: return launch_decode_sk_dg<T, D, 4>(a, kmap, vmap, stream);
    case 8: return launch_decode_sk_dg<T, D, 8>(a, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_decode_sk_t(const SkArgs& a, int head_dim, int gpad, const CUtensorMap* kmap,
                               const CUtensorMap* vmap, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_decode_sk_d<T, 64>(a, gpad, kmap, vmap, stream);
    case 128: return launch_decode_sk_d<T, 128>(a, gpad, kmap, vmap, stream);
    case 256: return launch_decode_sk_d<T, 256>(a, gpad, kmap, vmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
