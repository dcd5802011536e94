// Placement of the pinned host store on the GPU's NUMA node.
//
// The recall (the UVA gather) reads the host store over the GPU's host link at
// every decode step; on a host with several memory nodes (two Grace dies, or a
// multi-socket server) a store on another node than the GPU's own adds a hop on
// the very link the recall is bound by. nosa_create therefore binds the store's
// pages to the GPU's node (a preferred policy: the kernel falls back to other
// nodes rather than fail) before pinning them. With one memory node, or when
// the GPU's node is unknown, has no memory or is not allowed to this process,
// nothing is bound and the store is an ordinary cudaHostAlloc.
#include "nosa.h"
#include "nosa_internal.cuh"

#include <sys/mman.h>
#include <sys/syscall.h>
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

// Pinned, mapped host memory of `bytes`: bound (preferred) to `node` and then
// registered, or a plain cudaHostAlloc when node < 0 or binding is refused.
// *registered tells host_store_free which way it was made.
cudaError_t host_store_alloc(size_t bytes, int node, void** out, bool* registered) {
  *out = nullptr;
  *registered = false;
  if (node >= 0 && node < 1024) {
    void* p = mmap(nullptr, bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (p != MAP_FAILED) {
      unsigned long mask[1024 / (8 * sizeof(unsigned long))] = {0};
      mask[node / (8 * sizeof(unsigned long))] |= 1UL << (node % (8 * sizeof(unsigned long)));
      const long r = syscall(SYS_mbind, p, bytes, 1 /* MPOL_PREFERRED */, mask, 1024UL, 0U);
      if (r == 0 &&
          cudaHostRegister(p, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable) == cudaSuccess) {
        *out = p;
        *registered = true;
        return cudaSuccess;
      }
      cudaGetLastError();
      munmap(p, bytes);
    }
  }
  return cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
}

void host_store_free(void* p, size_t bytes, bool registered) {
  if (p == nullptr) return;
  if (registered) {
    cudaHostUnregister(p);
    munmap(p, bytes);
  } else {
    cudaFreeHost(p);
  }
}

}  // namespace nosa
