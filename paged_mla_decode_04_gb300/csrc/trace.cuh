// Optional event trace of the decode kernel's roles, compiled in only when
// the library is built with -DMLA_TRACE (the default build has none of it).
// Each role of each CTA appends records (SM clock, event, tile) to its own
// slice of a device buffer through its own Tracer; mla_trace_read copies the
// buffer to the host and clears it. One writer per slice (lane 0 of the
// role's warp), so no atomics.
#pragma once

#include <stdint.h>

namespace mla {

enum TraceEvent : uint32_t {
  kEvKernelStart = 1,   // kernel entry
  kEvSetupDone,         // barriers, TMEM and the plan read
  kEvKernelEnd,         // role loop left
  kEvSlotAcquired,      // producer: ring slot free for tile g
  kEvTileIssued,        // producer: TMA copies of tile g issued
  kEvQkTileReady,       // QK issuer: tile g landed
  kEvQkSFree,           // QK issuer: S buffer free for tile g
  kEvQkIssued,          // QK issuer: QK of tile g issued
  kEvSmSFull,           // softmax: S of tile g complete
  kEvSmSent,            // softmax: partial scores of tile g sent to the peer
  kEvSmXFull,           // softmax: the peer's partial scores of tile g landed
  kEvSmComputed,        // softmax: P of tile g in registers
  kEvSmPvDone,          // softmax: PV of the tile before g complete
  kEvSmOFixed,          // softmax: P of tile g in TMEM, O rescaled
  kEvSmItemStore,       // softmax: epilogue of the item ending at tile g begins
  kEvSmItemStored,      // softmax: epilogue done
  kEvPvOFixed,          // PV issuer: P of tile g ready
  kEvPvIssued,          // PV issuer: PV of tile g issued
  kEvQLoaded,           // QK issuer: q of the item ending before tile g copied to TMEM
  kEvSmXRead,           // softmax: the peer's partials of tile g read and released
  kEvSmPair,            // softmax: the row max of tile g shared with the row's other warp
  kEvGlobalStart,       // kernel entry, global timer (ns) instead of the SM clock
  kEvGlobalEnd,         // every role done (before TMEM release), global timer
  kEvGlobalExit,        // after the final cluster barrier, global timer
};

constexpr int kTraceRoles = 6;     // producer, QK, PV, softmax (first warp), softmax (last warp), spare
constexpr int kTraceCap = 2048;    // records per role per CTA
constexpr int kTraceCtas = 160;

}  // namespace mla

#ifdef MLA_TRACE
namespace mla {
__device__ uint64_t g_trace[kTraceCtas][kTraceRoles][kTraceCap];
__device__ uint32_t g_trace_n[kTraceCtas][kTraceRoles];

// One role's writer. Record: bits 0-39 SM clock, 40-47 event, 48-63 tile.
// The count lives in a register and is published with every record (a
// store only: reading it back from global memory would put an L2 round trip
// on every event).
struct Tracer {
  uint32_t n = 0;
  __device__ __forceinline__ void operator()(int role, uint32_t ev, uint32_t tile) {
    const uint32_t cta = blockIdx.x;
    if (cta >= kTraceCtas || n >= kTraceCap) return;
    uint64_t t;
    if (ev >= kEvGlobalStart) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    else t = clock64();
    g_trace[cta][role][n] = (t & 0xFFFFFFFFFFull) | (static_cast<uint64_t>(ev & 0xFF) << 40) |
                            (static_cast<uint64_t>(tile & 0xFFFF) << 48);
    g_trace_n[cta][role] = ++n;
  }
};
}  // namespace mla
#define MLA_TRACER(name) ::mla::Tracer name
#define MLA_TRACE_EVENT(tracer, role, ev, tile) (tracer)((role), (ev), (tile))
#else
#define MLA_TRACER(name) struct {} name
#define MLA_TRACE_EVENT(tracer, role, ev, tile) ((void)0)
#endif
