// Builds the library's device-side Philox4x32-10 (csrc/philox.cuh) as plain
// host C++ so that a test can compare it with the oracle's own, separately
// written generator without a GPU (tests/test_device_philox_on_host.py).
//
// The device code calls __umulhi, the high 32 bits of a 32 x 32-bit product;
// here it is that definition written out.  __device__ and __forceinline__ are
// defined away.
//
// usage: device_philox_host_driver kat   < "c0 c1 c2 c3 k0 k1" hex lines -> word 0 (hex)
//        device_philox_host_driver grid in.bin out.bin
//          in.bin: records {uint64 seed, uint64 seq, uint32 pos, uint32 draw}
//          out.bin: one float32 uniform per record
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

static inline uint32_t __umulhi(uint32_t a, uint32_t b) {
  return static_cast<uint32_t>((static_cast<uint64_t>(a) * b) >> 32);
}
#define __device__
#define __forceinline__ inline
#include "philox.cuh"

struct Request {
  uint64_t seed, seq;
  uint32_t pos, draw;
};
static_assert(sizeof(Request) == 24, "record layout");

int main(int argc, char** argv) {
  if (argc >= 2 && std::strcmp(argv[1], "kat") == 0) {
    unsigned c[4], k[2];
    while (std::scanf("%x %x %x %x %x %x", &c[0], &c[1], &c[2], &c[3], &k[0], &k[1]) == 6)
      std::printf("%08x\n", sv::philox4x32_10_word0(c[0], c[1], c[2], c[3], k[0], k[1]));
    return 0;
  }
  if (argc == 4 && std::strcmp(argv[1], "grid") == 0) {
    std::FILE* in = std::fopen(argv[2], "rb");
    if (!in) return 2;
    std::vector<Request> req;
    Request r;
    while (std::fread(&r, sizeof r, 1, in) == 1) req.push_back(r);
    std::fclose(in);
    std::vector<float> out(req.size());
    for (size_t i = 0; i < req.size(); ++i)
      out[i] = sv::philox_uniform(req[i].seed, req[i].seq, req[i].pos, req[i].draw);
    std::FILE* o = std::fopen(argv[3], "wb");
    if (!o) return 2;
    const size_t n = std::fwrite(out.data(), sizeof(float), out.size(), o);
    std::fclose(o);
    return n == out.size() ? 0 : 3;
  }
  std::fprintf(stderr, "usage: %s kat | grid in.bin out.bin\n", argv[0]);
  return 1;
}
