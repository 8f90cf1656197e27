// One device virtual range holding a VRAM head and a host-memory tail, with
// an optional second range that aliases the same head pages followed by a
// VRAM staging buffer (llama.cpp PR #319 "tiered KV cache (--kv-vram-cells):
// VRAM head, pinned-host tail in one VMM range", the tier buffer and its
// review: the Linux driver takes CU_MEM_LOCATION_TYPE_HOST_NUMA with the id
// CU_DEVICE_ATTRIBUTE_HOST_NUMA_ID, not CU_MEM_LOCATION_TYPE_HOST).
//
// The driver's virtual-memory calls are fetched once through the runtime
// (cudaGetDriverEntryPointByVersion), so the library links no libcuda.  Every
// range a tier maps is recorded, so that the rest of the library knows which
// addresses are host-backed (vmm_host_backed): those are read with plain
// loads only, never with cp.async or TMA.
#include <cuda.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvo_internal.cuh"

namespace kvo {
namespace {

struct Drv {
  CUresult (*mem_create)(CUmemGenericAllocationHandle *, size_t, const CUmemAllocationProp *, unsigned long long);
  CUresult (*mem_release)(CUmemGenericAllocationHandle);
  CUresult (*addr_reserve)(CUdeviceptr *, size_t, size_t, CUdeviceptr, unsigned long long);
  CUresult (*addr_free)(CUdeviceptr, size_t);
  CUresult (*mem_map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long);
  CUresult (*mem_unmap)(CUdeviceptr, size_t);
  CUresult (*set_access)(CUdeviceptr, size_t, const CUmemAccessDesc *, size_t);
  CUresult (*granularity)(size_t *, const CUmemAllocationProp *, CUmemAllocationGranularity_flags);
  CUresult (*dev_attr)(int *, CUdevice_attribute, CUdevice);
  CUresult (*dev_get)(CUdevice *, int);
  CUresult (*ptr_attr)(void *, CUpointer_attribute, CUdeviceptr);   // optional: range queries
  bool ok = false;
};

const Drv &drv() {
  static Drv d;
  static std::once_flag once;
  std::call_once(once, [] {
    auto get = [](const char *name, void **fn) {
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      if (cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !*fn) {
        cudaGetLastError();
        *fn = nullptr;
        return false;
      }
      return true;
    };
    bool ok = true;
    ok &= get("cuMemCreate", (void **)&d.mem_create);
    ok &= get("cuMemRelease", (void **)&d.mem_release);
    ok &= get("cuMemAddressReserve", (void **)&d.addr_reserve);
    ok &= get("cuMemAddressFree", (void **)&d.addr_free);
    ok &= get("cuMemMap", (void **)&d.mem_map);
    ok &= get("cuMemUnmap", (void **)&d.mem_unmap);
    ok &= get("cuMemSetAccess", (void **)&d.set_access);
    ok &= get("cuMemGetAllocationGranularity", (void **)&d.granularity);
    ok &= get("cuDeviceGetAttribute", (void **)&d.dev_attr);
    ok &= get("cuDeviceGet", (void **)&d.dev_get);
    d.ok = ok;
    get("cuPointerGetAttribute", (void **)&d.ptr_attr);
  });
  return d;
}

CUmemAllocationProp prop_for(int device, bool host, int numa_id) {
  CUmemAllocationProp p;
  std::memset(&p, 0, sizeof p);
  p.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  p.location.type = host ? CU_MEM_LOCATION_TYPE_HOST_NUMA : CU_MEM_LOCATION_TYPE_DEVICE;
  p.location.id = host ? numa_id : device;
  return p;
}

struct Tier {
  int device = 0;
  CUdeviceptr base = 0, alias = 0;
  size_t head = 0, tail = 0, stage = 0;
  CUmemGenericAllocationHandle h_head = 0, h_tail = 0, h_stage = 0;
  bool head_ok = false, tail_ok = false, stage_ok = false;
  bool base_mapped_head = false, base_mapped_tail = false, alias_mapped_head = false, alias_mapped_stage = false;
};

void release(Tier *t) {
  const Drv &d = drv();
  if (t->alias_mapped_stage) d.mem_unmap(t->alias + t->head, t->stage);
  if (t->alias_mapped_head) d.mem_unmap(t->alias, t->head);
  if (t->base_mapped_tail) d.mem_unmap(t->base + t->head, t->tail);
  if (t->base_mapped_head) d.mem_unmap(t->base, t->head);
  if (t->alias) d.addr_free(t->alias, t->head + t->stage);
  if (t->base) d.addr_free(t->base, t->head + t->tail);
  if (t->stage_ok) d.mem_release(t->h_stage);
  if (t->tail_ok) d.mem_release(t->h_tail);
  if (t->head_ok) d.mem_release(t->h_head);
  delete t;
}

int drv_status(CUresult r, const char *what) {
  if (r == CUDA_SUCCESS) return KVO_OK;
  if (r == CUDA_ERROR_NOT_SUPPORTED) return fail(KVO_ERR_UNSUPPORTED, "%s: not supported (CUresult %d)", what, (int)r);
  return fail(KVO_ERR_CUDA, "%s failed (CUresult %d)", what, (int)r);
}

// Keeps the caller's current device: the calls below act on `device`.
struct DeviceScope {
  int prev = -1;
  explicit DeviceScope(int device) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    cudaSetDevice(device);
    cudaFree(nullptr);                       // the primary context exists from here on
  }
  ~DeviceScope() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

size_t round_up(size_t x, size_t g) { return (x + g - 1) / g * g; }

// The host NUMA node the device reports (node 0 where the host has none).
int host_numa_of(const Drv &d, int device) {
  CUdevice dev = 0;
  int numa = -1;
  if (d.dev_get(&dev, device) != CUDA_SUCCESS ||
      d.dev_attr(&numa, CU_DEVICE_ATTRIBUTE_HOST_NUMA_ID, dev) != CUDA_SUCCESS)
    numa = -1;
  return numa < 0 ? 0 : numa;
}

// The mapped ranges of the live tiers: [lo, hi), host-backed or not.
struct Range {
  uintptr_t lo, hi;
  int host;
  const Tier *owner;
};
std::mutex reg_mu;
std::vector<Range> &registry() {
  static std::vector<Range> r;
  return r;
}

void register_tier(const Tier *t) {
  std::lock_guard<std::mutex> lock(reg_mu);
  auto &r = registry();
  r.push_back({(uintptr_t)t->base, (uintptr_t)(t->base + t->head), 0, t});
  r.push_back({(uintptr_t)(t->base + t->head), (uintptr_t)(t->base + t->head + t->tail), 1, t});
  if (t->stage) r.push_back({(uintptr_t)t->alias, (uintptr_t)(t->alias + t->head + t->stage), 0, t});
}

void unregister_tier(const Tier *t) {
  std::lock_guard<std::mutex> lock(reg_mu);
  auto &r = registry();
  for (size_t i = 0; i < r.size();)
    if (r[i].owner == t) r.erase(r.begin() + (long)i);
    else ++i;
}

}  // namespace

int vmm_host_backed(const void *p, uintptr_t *range_end) {
  std::lock_guard<std::mutex> lock(reg_mu);
  const uintptr_t a = (uintptr_t)p;
  for (const Range &r : registry())
    if (a >= r.lo && a < r.hi) {
      if (range_end) *range_end = r.hi;
      return r.host;
    }
  return -1;
}

bool alloc_range(const void *p, uintptr_t *lo, uintptr_t *hi) {
  const Drv &d = drv();
  if (!d.ptr_attr) return false;
  CUdeviceptr start = 0;
  size_t size = 0;
  if (d.ptr_attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, (CUdeviceptr)(uintptr_t)p) != CUDA_SUCCESS ||
      d.ptr_attr(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, (CUdeviceptr)(uintptr_t)p) != CUDA_SUCCESS)
    return false;
  *lo = (uintptr_t)start;
  *hi = (uintptr_t)start + size;
  return *lo <= (uintptr_t)p && (uintptr_t)p < *hi;
}

}  // namespace kvo

using namespace kvo;

extern "C" int kvo_vmm_granularity(int device, size_t *bytes) {
  clear_error();
  if (!bytes) return fail(KVO_ERR_ARG, "kvo_vmm_granularity: NULL bytes");
  *bytes = 0;
  const Drv &d = drv();
  if (!d.ok) return fail(KVO_ERR_UNSUPPORTED, "kvo_vmm_granularity: driver virtual-memory calls unavailable");
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) {
    cudaGetLastError();
    return fail(KVO_ERR_ARG, "kvo_vmm_granularity: no device %d", device);
  }
  DeviceScope scope(device);
  const int numa = host_numa_of(d, device);
  size_t g_dev = 0, g_host = 0;
  const CUmemAllocationProp pd = prop_for(device, false, 0), ph = prop_for(device, true, numa);
  int e = drv_status(d.granularity(&g_dev, &pd, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED), "cuMemGetAllocationGranularity");
  if (!e) e = drv_status(d.granularity(&g_host, &ph, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED), "cuMemGetAllocationGranularity");
  if (e) return e;
  *bytes = g_dev > g_host ? g_dev : g_host;
  return KVO_OK;
}

extern "C" int kvo_vmm_tier_create(int device, size_t head_bytes, size_t tail_bytes, size_t stage_bytes,
                                   void **base, void **alias, size_t *head_mapped, size_t *tail_mapped,
                                   size_t *stage_mapped, void **tier) {
  clear_error();
  const char *fn = "kvo_vmm_tier_create";
  if (!base || !tier) return fail(KVO_ERR_ARG, "%s: NULL base or tier", fn);
  *base = nullptr;
  *tier = nullptr;
  if (alias) *alias = nullptr;
  if (head_bytes == 0 || tail_bytes == 0) return fail(KVO_ERR_ARG, "%s: head and tail must both be non-empty", fn);
  if (stage_bytes && !alias) return fail(KVO_ERR_ARG, "%s: stage_bytes > 0 needs an alias output", fn);
  size_t g = 0;
  int e = kvo_vmm_granularity(device, &g);
  if (e) return e;
  const Drv &d = drv();
  DeviceScope scope(device);
  const int numa = host_numa_of(d, device);

  Tier *t = new Tier;
  t->device = device;
  t->head = round_up(head_bytes, g);
  t->tail = round_up(tail_bytes, g);
  t->stage = stage_bytes ? round_up(stage_bytes, g) : 0;
  const CUmemAllocationProp pd = prop_for(device, false, 0), ph = prop_for(device, true, numa);
  CUmemAccessDesc acc;
  std::memset(&acc, 0, sizeof acc);
  acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  acc.location.id = device;
  acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;

  e = drv_status(d.mem_create(&t->h_head, t->head, &pd, 0), "cuMemCreate (VRAM head)");
  t->head_ok = !e;
  if (!e) {
    e = drv_status(d.mem_create(&t->h_tail, t->tail, &ph, 0), "cuMemCreate (host NUMA tail)");
    t->tail_ok = !e;
  }
  if (!e && t->stage) {
    e = drv_status(d.mem_create(&t->h_stage, t->stage, &pd, 0), "cuMemCreate (staging)");
    t->stage_ok = !e;
  }
  if (!e) e = drv_status(d.addr_reserve(&t->base, t->head + t->tail, g, 0, 0), "cuMemAddressReserve");
  if (!e) {
    e = drv_status(d.mem_map(t->base, t->head, 0, t->h_head, 0), "cuMemMap (head)");
    t->base_mapped_head = !e;
  }
  if (!e) {
    e = drv_status(d.mem_map(t->base + t->head, t->tail, 0, t->h_tail, 0), "cuMemMap (tail)");
    t->base_mapped_tail = !e;
  }
  if (!e) e = drv_status(d.set_access(t->base, t->head, &acc, 1), "cuMemSetAccess (head)");
  if (!e) e = drv_status(d.set_access(t->base + t->head, t->tail, &acc, 1), "cuMemSetAccess (tail)");
  if (!e && t->stage) {
    e = drv_status(d.addr_reserve(&t->alias, t->head + t->stage, g, 0, 0), "cuMemAddressReserve (alias)");
    if (!e) {
      e = drv_status(d.mem_map(t->alias, t->head, 0, t->h_head, 0), "cuMemMap (alias head)");
      t->alias_mapped_head = !e;
    }
    if (!e) {
      e = drv_status(d.mem_map(t->alias + t->head, t->stage, 0, t->h_stage, 0), "cuMemMap (alias staging)");
      t->alias_mapped_stage = !e;
    }
    if (!e) e = drv_status(d.set_access(t->alias, t->head + t->stage, &acc, 1), "cuMemSetAccess (alias)");
  }
  if (e) {
    release(t);
    return e;
  }
  register_tier(t);
  *base = (void *)t->base;
  if (alias) *alias = t->stage ? (void *)t->alias : nullptr;
  if (head_mapped) *head_mapped = t->head;
  if (tail_mapped) *tail_mapped = t->tail;
  if (stage_mapped) *stage_mapped = t->stage;
  *tier = t;
  return KVO_OK;
}

extern "C" int kvo_vmm_tier_destroy(void *tier) {
  clear_error();
  if (!tier) return KVO_OK;
  Tier *t = (Tier *)tier;
  DeviceScope scope(t->device);
  if (cudaDeviceSynchronize() != cudaSuccess) {   // no kernel may still read the range
    cudaGetLastError();
    return fail(KVO_ERR_CUDA, "kvo_vmm_tier_destroy: device synchronisation failed");
  }
  unregister_tier(t);
  release(t);
  return KVO_OK;
}
