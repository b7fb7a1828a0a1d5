// Host-side helpers of libkvm.so shared between translation units:
// configuration validation, workspace layout and the data-independent
// growth schedule.  Defined in kvm_api.cu.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/kvm.h"
#include "kvm_internal.cuh"

namespace kvm {
namespace host {

constexpr size_t ALIGN = 256;

// Byte offsets of every array inside a layer's workspace.
struct Layout {
    size_t sum_k, sum_v, counts, rho, simdir, view_k, view_v;
    size_t ring_k, ring_v, ring_g, ring_kr, snap_k, snap_v, rope, sched, status, total;
};

extern thread_local std::string g_err;

size_t align_up(size_t x);
int64_t n_events_for(const kvm_config& c, int64_t N);
int64_t capacity(const kvm_config& c, int64_t t);
Sched event_sched(const kvm_config& c, int64_t first_pos, int64_t n, int64_t t);
bool validate(const kvm_config* c, std::string& why);
Layout layout_of(const kvm_config& c);

}  // namespace host
}  // namespace kvm
