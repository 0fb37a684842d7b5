// Checkpoint files of the training state: the fp32 master weights and the
// RMSProp state, in the parameter packing order, and a step count.  The GPipe
// technical review ("Limitations 6") notes that GPipe has no fault tolerance
// and that later systems recover through checkpoints; its synchronous step makes a
// resumed run identical to an uninterrupted one, since the state between
// steps is exactly (w, v) (the gradient buffer is zero after each update).
//
// Layout (little-endian): "GPIPECK1", u32 version (1), u32 kind, L, d,
// heads, seq, vocab, dtype, u64 parameter count, u64 layout fingerprint
// (FNV-1a over the shape fields and every layer's FFN width), u64 step,
// u64 payload checksum (FNV-1a over the bytes that follow), then P floats of
// weights and P floats of RMSProp state.  Written to path.tmp, flushed to the
// disk (fsync), renamed over path, and the directory flushed too: after a
// crash or power loss at any point, path holds either the previous complete
// checkpoint or the new one, never a renamed file whose data did not land.
#include <fcntl.h>
#include <unistd.h>

#include <cerrno>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/gpipe.h"
#include "context_info.h"

namespace {

constexpr char kMagic[8] = {'G', 'P', 'I', 'P', 'E', 'C', 'K', '1'};
constexpr uint32_t kVersion = 1;
constexpr uint64_t kFnvOffset = 1469598103934665603ull, kFnvPrime = 1099511628211ull;

uint64_t fnv1a(uint64_t h, const void* data, size_t n) {
  const unsigned char* p = static_cast<const unsigned char*>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= kFnvPrime;
  }
  return h;
}

struct Header {
  uint32_t version, kind, L, d, heads, seq, vocab, dtype;
  uint64_t params, layout, step, checksum;
};
constexpr size_t kHeaderBytes = 8 + 8 * 4 + 4 * 8;

void put32(std::vector<unsigned char>& b, uint32_t v) {
  for (int i = 0; i < 4; ++i) b.push_back(static_cast<unsigned char>(v >> (8 * i)));
}
void put64(std::vector<unsigned char>& b, uint64_t v) {
  for (int i = 0; i < 8; ++i) b.push_back(static_cast<unsigned char>(v >> (8 * i)));
}
uint32_t get32(const unsigned char* p) {
  uint32_t v = 0;
  for (int i = 0; i < 4; ++i) v |= static_cast<uint32_t>(p[i]) << (8 * i);
  return v;
}
uint64_t get64(const unsigned char* p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; ++i) v |= static_cast<uint64_t>(p[i]) << (8 * i);
  return v;
}

// The header this context would write (step and checksum left 0).
Header expected(const gpipe_ctx* c) {
  gp::Dims dm{};
  int L = 0;
  std::vector<int> ffn;
  size_t P = 0;
  gp::describe_context(c, &dm, &L, &ffn, &P);
  Header h{kVersion, static_cast<uint32_t>(dm.kind), static_cast<uint32_t>(L), static_cast<uint32_t>(dm.d),
           static_cast<uint32_t>(dm.heads), static_cast<uint32_t>(dm.seq), static_cast<uint32_t>(dm.vocab),
           static_cast<uint32_t>(dm.dtype), P, 0, 0, 0};
  std::vector<unsigned char> shape;
  for (uint32_t v : {h.kind, h.L, h.d, h.heads, h.seq, h.vocab, h.dtype}) put32(shape, v);
  for (int f : ffn) put32(shape, static_cast<uint32_t>(f));
  h.layout = fnv1a(kFnvOffset, shape.data(), shape.size());
  return h;
}

int io_fail(const gpipe_ctx* c, const std::string& msg) {
  return gp::context_fail(const_cast<gpipe_ctx*>(c), GPIPE_ERR_IO, msg.c_str());
}

// Flush the directory that holds path, so that a rename inside it is durable.
bool sync_parent_dir(const std::string& path) {
  const size_t slash = path.find_last_of('/');
  const std::string dir = slash == std::string::npos ? "." : (slash == 0 ? "/" : path.substr(0, slash));
  const int fd = open(dir.c_str(), O_RDONLY | O_DIRECTORY);
  if (fd < 0) return false;
  const bool ok = fsync(fd) == 0;
  return (close(fd) == 0) && ok;
}

}  // namespace

extern "C" {

int gpipe_checkpoint_write(const gpipe_ctx* c, const char* path, const float* params, const float* rms_v,
                           uint64_t step) {
  if (!c || !path || !params || !rms_v) return GPIPE_ERR_INVALID_ARG;
  Header h = expected(c);
  const size_t bytes = h.params * sizeof(float);
  h.step = step;
  h.checksum = fnv1a(fnv1a(kFnvOffset, params, bytes), rms_v, bytes);
  std::vector<unsigned char> head(kMagic, kMagic + 8);
  for (uint32_t v : {h.version, h.kind, h.L, h.d, h.heads, h.seq, h.vocab, h.dtype}) put32(head, v);
  for (uint64_t v : {h.params, h.layout, h.step, h.checksum}) put64(head, v);
  const std::string tmp = std::string(path) + ".tmp";
  FILE* f = std::fopen(tmp.c_str(), "wb");
  if (!f) return io_fail(c, "cannot open " + tmp + ": " + std::strerror(errno));
  bool ok = std::fwrite(head.data(), 1, head.size(), f) == head.size() &&
            std::fwrite(params, 1, bytes, f) == bytes && std::fwrite(rms_v, 1, bytes, f) == bytes;
  // the data reaches the disk before the rename can make it the checkpoint
  ok = ok && std::fflush(f) == 0 && fsync(fileno(f)) == 0;
  ok = (std::fclose(f) == 0) && ok;
  if (!ok || std::rename(tmp.c_str(), path) != 0) {
    std::remove(tmp.c_str());
    return io_fail(c, std::string("cannot write ") + path);
  }
  if (!sync_parent_dir(path)) return io_fail(c, std::string("cannot flush the directory of ") + path);
  return GPIPE_OK;
}

int gpipe_checkpoint_read(const gpipe_ctx* c, const char* path, float* params, float* rms_v, uint64_t* step) {
  if (!c || !path || !params || !rms_v) return GPIPE_ERR_INVALID_ARG;
  const Header want = expected(c);
  FILE* f = std::fopen(path, "rb");
  if (!f) return io_fail(c, std::string("cannot open ") + path + ": " + std::strerror(errno));
  unsigned char head[kHeaderBytes];
  if (std::fread(head, 1, kHeaderBytes, f) != kHeaderBytes || std::memcmp(head, kMagic, 8) != 0) {
    std::fclose(f);
    return io_fail(c, std::string(path) + " is not a checkpoint of this library");
  }
  Header h{};
  uint32_t* f32[] = {&h.version, &h.kind, &h.L, &h.d, &h.heads, &h.seq, &h.vocab, &h.dtype};
  for (int i = 0; i < 8; ++i) *f32[i] = get32(head + 8 + 4 * i);
  uint64_t* f64[] = {&h.params, &h.layout, &h.step, &h.checksum};
  for (int i = 0; i < 4; ++i) *f64[i] = get64(head + 40 + 8 * i);
  if (h.version != kVersion) {
    std::fclose(f);
    return io_fail(c, "unsupported checkpoint version " + std::to_string(h.version));
  }
  if (h.params != want.params || h.layout != want.layout) {
    std::fclose(f);
    return io_fail(c, std::string(path) + " was written for a different model (shape or parameter count)");
  }
  const size_t bytes = h.params * sizeof(float);
  // read into staging so a bad file leaves the caller's buffers untouched
  std::vector<float> w(h.params), v(h.params);
  const bool full = std::fread(w.data(), 1, bytes, f) == bytes && std::fread(v.data(), 1, bytes, f) == bytes;
  const bool at_end = std::fgetc(f) == EOF;
  std::fclose(f);
  if (!full || !at_end) return io_fail(c, std::string(path) + " has the wrong length");
  if (fnv1a(fnv1a(kFnvOffset, w.data(), bytes), v.data(), bytes) != h.checksum)
    return io_fail(c, std::string(path) + " is corrupt (checksum mismatch)");
  std::memcpy(params, w.data(), bytes);
  std::memcpy(rms_v, v.data(), bytes);
  if (step) *step = h.step;
  return GPIPE_OK;
}

}  // extern "C"
