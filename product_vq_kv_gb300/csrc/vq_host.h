// vq_host.h -- host helpers shared by the library's translation units
// (internal; not part of the C ABI).
#pragma once

// Streaming multiprocessors of the current device, cached per device; 0 if
// there is no usable device.
int vqh_device_sms();
