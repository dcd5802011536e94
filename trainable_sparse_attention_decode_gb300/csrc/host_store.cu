// Placement of the pinned host store on the GPU's NUMA node.
//
// The recall (the UVA gather) reads the host store over the GPU's host link at
// every decode step; on a host with several memory nodes (two Grace dies, or a
// multi-socket server) a store on another node than the GPU's own adds a hop on
// the very link the recall is bound by. nosa_create therefore binds the store's
// pages to the GPU's node (a preferred policy: the kernel falls back to other
// nodes rather than fail) before pinning them. With one memory node, or when
// the GPU's node is unknown, has no memory or is not allowed to this process,
// nothing is bound. A store of 1 GiB or more, bound or not, is laid out in
// pinned transparent huge pages (host_store_alloc).
#include "nosa.h"
#include "nosa_internal.cuh"

#include <sys/mman.h>
#include <sys/syscall.h>
#include <sys/uio.h>
#include <unistd.h>

#include <cctype>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

extern "C" int32_t nosa_numa_choose(int32_t gpu_node, const int32_t* mem_nodes, int32_t n_mem,
                                    const int32_t* allowed, int32_t n_allowed) {
  if (gpu_node < 0 || n_mem < 2 || mem_nodes == nullptr || allowed == nullptr) return -1;
  bool has_mem = false, ok = false;
  for (int i = 0; i < n_mem; ++i) has_mem |= (mem_nodes[i] == gpu_node);
  for (int i = 0; i < n_allowed; ++i) ok |= (allowed[i] == gpu_node);
  return (has_mem && ok) ? gpu_node : -1;
}

namespace nosa {
namespace {

std::string read_small(const std::string& path) {
  FILE* f = std::fopen(path.c_str(), "r");
  if (!f) return "";
  char buf[4096];
  const size_t n = std::fread(buf, 1, sizeof(buf) - 1, f);
  std::fclose(f);
  buf[n] = 0;
  return std::string(buf);
}

// "0-3,8,10-11" -> {0,1,2,3,8,10,11}
std::vector<int> parse_list(const std::string& s) {
  std::vector<int> out;
  size_t i = 0;
  while (i < s.size()) {
    if (!std::isdigit((unsigned char)s[i])) { ++i; continue; }
    int a = 0;
    while (i < s.size() && std::isdigit((unsigned char)s[i])) a = a * 10 + (s[i++] - '0');
    int b = a;
    if (i < s.size() && s[i] == '-') {
      ++i;
      b = 0;
      while (i < s.size() && std::isdigit((unsigned char)s[i])) b = b * 10 + (s[i++] - '0');
    }
    for (int x = a; x <= b && x - a < 4096; ++x) out.push_back(x);
  }
  return out;
}

}  // namespace

// Node to bind the host store of `device` to, or -1 (see nosa_numa_choose).
int host_store_node(int device) {
  char bus[64] = {0};
  if (cudaDeviceGetPCIBusId(bus, sizeof(bus), device) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  for (char* c = bus; *c; ++c) *c = (char)std::tolower((unsigned char)*c);
  const std::string n = read_small(std::string("/sys/bus/pci/devices/") + bus + "/numa_node");
  if (n.empty()) return -1;
  const int gpu_node = std::atoi(n.c_str());
  // nodes with CPUs and memory (a GPU's own memory may show as a node without CPUs)
  std::vector<int> mem_nodes;
  for (int node : parse_list(read_small("/sys/devices/system/node/has_memory"))) {
    const std::string cpus =
        read_small("/sys/devices/system/node/node" + std::to_string(node) + "/cpulist");
    if (!parse_list(cpus).empty()) mem_nodes.push_back(node);
  }
  std::vector<int> allowed;
  const std::string status = read_small("/proc/self/status");
  const size_t at = status.find("Mems_allowed_list:");
  if (at != std::string::npos)
    allowed = parse_list(status.substr(at + 18, status.find('\n', at) - at - 18));
  return nosa_numa_choose(gpu_node, mem_nodes.data(), (int)mem_nodes.size(), allowed.data(),
                          (int)allowed.size());
}

namespace {

// madvise advice values of Linux 5.14 (populate for writing) and 6.1 (collapse into
// huge pages); older kernels answer EINVAL and the call does nothing.
constexpr int kMadvPopulateWrite = 23;
constexpr int kMadvCollapse = 25;

// io_uring system calls (the same numbers on every architecture since Linux 5.1).
#ifdef SYS_io_uring_setup
constexpr long kSysUringSetup = SYS_io_uring_setup;
constexpr long kSysUringRegister = SYS_io_uring_register;
#else
constexpr long kSysUringSetup = 425;
constexpr long kSysUringRegister = 427;
#endif

// The size of a transparent huge page (the page-middle-directory size: 2 MB with
// 4 KB base pages, 512 MB with 64 KB ones), or 0 where the kernel has none or
// they are switched off ("[never]": MADV_HUGEPAGE would then do nothing).
size_t thp_size() {
  if (std::FILE* e = std::fopen("/sys/kernel/mm/transparent_hugepage/enabled", "r")) {
    char mode[128] = {0};
    const size_t n = std::fread(mode, 1, sizeof(mode) - 1, e);
    std::fclose(e);
    mode[n] = 0;
    if (std::strstr(mode, "[never]") != nullptr) return 0;
  }
  std::FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r");
  if (f == nullptr) return 0;
  unsigned long long v = 0;
  if (std::fscanf(f, "%llu", &v) != 1) v = 0;
  std::fclose(f);
  return (v & (v - 1)) == 0 ? (size_t)v : 0;  // a power of two, or nothing
}

// An anonymous mapping of `len` bytes that starts on a multiple of `align` (a
// power of two), or nullptr.
void* map_aligned(size_t len, size_t align) {
  void* raw = mmap(nullptr, len + align, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS,
                   -1, 0);
  if (raw == MAP_FAILED) return nullptr;
  const uintptr_t r = reinterpret_cast<uintptr_t>(raw);
  const uintptr_t a = (r + align - 1) & ~(uintptr_t)(align - 1);
  if (a > r) munmap(raw, a - r);
  munmap(reinterpret_cast<void*>(a + len), r + align - a);
  return reinterpret_cast<void*>(a);
}

// Pins [p, p + len) for as long as the returned descriptor stays open (-1: not
// pinned). The range is registered as the fixed buffers of an io_uring instance,
// which holds long-term pins on its pages: the kernel can then neither migrate
// nor split them while the GPU reads them (cudaHostRegister does not prevent
// either where the GPU reaches host memory through the host's own page tables).
// Buffers of 1 GiB at most each. Needs CAP_IPC_LOCK or a locked-memory limit
// above `len`; the descriptor is close-on-exec.
int pin_long_term(void* p, size_t len) {
  unsigned char params[120];  // struct io_uring_params, all zero: defaults
  std::memset(params, 0, sizeof(params));
  const long fd = syscall(kSysUringSetup, 1, params);
  if (fd < 0) return -1;
  const size_t gib = (size_t)1 << 30;
  std::vector<struct iovec> iov;
  for (size_t off = 0; off < len; off += gib) {
    struct iovec v;
    v.iov_base = static_cast<char*>(p) + off;
    v.iov_len = len - off < gib ? len - off : gib;
    iov.push_back(v);
  }
  const long r = syscall(kSysUringRegister, (int)fd, 0 /* IORING_REGISTER_BUFFERS */,
                         iov.data(), (unsigned)iov.size());
  if (r < 0) {
    close((int)fd);
    return -1;
  }
  return (int)fd;
}

// Whether this process may create io_uring instances at all (a seccomp filter or
// kernel.io_uring_disabled can forbid it); probed once, so that a store that needs
// the pin is not faulted in only to be thrown away.
bool uring_available() {
  static const bool ok = [] {
    unsigned char params[120];
    std::memset(params, 0, sizeof(params));
    const long fd = syscall(kSysUringSetup, 1, params);
    if (fd < 0) return false;
    close((int)fd);
    return true;
  }();
  return ok;
}

// Drops the pins of pin_long_term at once (closing the descriptor alone releases
// them only when the kernel tears the instance down, some time later).
void unpin(int fd) {
  if (fd < 0) return;
  syscall(kSysUringRegister, fd, 1 /* IORING_UNREGISTER_BUFFERS */, nullptr, 0U);
  close(fd);
}

// One registered anonymous mapping of at least `bytes`: aligned to and rounded up
// to `page`, bound (preferred) to `node` when node >= 0, advised into transparent
// huge pages when `huge`, faulted in (what came out small collapsed), pinned where
// pin_long_term can (not tried without `try_pin`), then registered with
// cudaHostRegister. Returns nullptr (and
// releases everything) when a step fails or when `need_pin` and the pin did not hold.
void* map_registered(size_t bytes, size_t page, int node, bool huge, bool need_pin,
                     bool try_pin, size_t* len_out, int* pin_fd) {
  *pin_fd = -1;
  const bool can_pin = try_pin && uring_available();
  if (need_pin && !can_pin) return nullptr;
  const size_t len = (bytes + page - 1) / page * page;
  void* p = map_aligned(len, page);
  if (p == nullptr) return nullptr;
  bool ok = true;
  if (node >= 0) {
    unsigned long mask[1024 / (8 * sizeof(unsigned long))] = {0};
    mask[node / (8 * sizeof(unsigned long))] |= 1UL << (node % (8 * sizeof(unsigned long)));
    ok = syscall(SYS_mbind, p, len, 1 /* MPOL_PREFERRED */, mask, 1024UL, 0U) == 0;
  }
  if (ok) {
    if (huge) madvise(p, len, MADV_HUGEPAGE);
    madvise(p, len, MADV_DONTFORK);  // a forked child never sees the store
    madvise(p, len, kMadvPopulateWrite);
    if (huge) madvise(p, len, kMadvCollapse);
    *pin_fd = can_pin ? pin_long_term(p, len) : -1;
    ok = !need_pin || *pin_fd >= 0;
  }
  if (ok && cudaHostRegister(p, len, cudaHostRegisterMapped | cudaHostRegisterPortable) ==
                cudaSuccess) {
    *len_out = len;
    return p;
  }
  cudaGetLastError();
  unpin(*pin_fd);
  *pin_fd = -1;
  munmap(p, len);
  return nullptr;
}

}  // namespace

// Pinned host memory of at least `bytes`, reachable by the device. *kind says how
// it was made (host_store_free needs it), *mapped its mapped length, *pin_fd the
// descriptor that holds its pages (-1: none):
//   kind 1: a mapping bound to `node` (node >= 0): in pinned transparent huge pages
//           for stores of 1 GiB or more; where the pin does not hold, in base pages
//           (pinned if it can be), as huge pages may be split under the GPU;
//   kind 2: an unbound mapping in transparent huge pages (stores of 1 GiB or more),
//           taken only when the pin holds;
//   kind 0: a plain cudaHostAlloc (everything else, and the fallback).
// Why the huge pages: the recall reads about 1 300 scattered blocks of the store
// per step, and with 64 KB pages their address translation, not the link, set the
// rate in most short runs on the GB300 machines (medians well above the link-bound
// step, up to 2.9x); with 512 MB pages every run kept the link's rate. Why the
// pins: without them the kernel split the huge pages of a running store now and
// then, and every step of that run took milliseconds. NOSA_HOST_HUGEPAGE=0 keeps
// the plain store (or the bound base-page mapping).
cudaError_t host_store_alloc(size_t bytes, int node, void** out, int* kind, size_t* mapped,
                             int* pin_fd, bool try_pin) {
  *pin_fd = -1;
  *out = nullptr;
  *kind = 0;
  *mapped = bytes;
  const char* g = std::getenv("NOSA_HOST_HUGEPAGE");
  const bool bind = node >= 0 && node < 1024;
  const size_t huge =
      (g == nullptr || std::atoi(g) != 0) && bytes >= ((size_t)1 << 30) ? thp_size() : 0;
  const size_t base = (size_t)sysconf(_SC_PAGESIZE);
  void* p = nullptr;
  if (huge != 0)
    p = map_registered(bytes, huge, bind ? node : -1, true, true, try_pin, mapped, pin_fd);
  if (p == nullptr && bind)
    p = map_registered(bytes, base, node, false, false, try_pin, mapped, pin_fd);
  if (p != nullptr) {
    *out = p;
    *kind = bind ? 1 : 2;
    return cudaSuccess;
  }
  *mapped = bytes;
  return cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
}

void host_store_free(void* p, size_t mapped, int kind, int pin_fd) {
  if (p == nullptr) return;
  if (kind == 1 || kind == 2) {
    cudaHostUnregister(p);
    unpin(pin_fd);
    munmap(p, mapped);
  } else {
    cudaFreeHost(p);
  }
}

}  // namespace nosa
