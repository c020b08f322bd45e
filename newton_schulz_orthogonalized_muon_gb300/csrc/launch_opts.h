// Per-call launch options of the element-wise kernels (host side).
#pragma once

namespace muon {

// Programmatic dependent launch for the element-wise kernels (preparation,
// norm, final apply) launched by this thread: on for small sets, where their
// launch latency shows between the short products; off for large ones,
// where an early-launched preparation's small CTAs sit beside a running
// GEMM's CTA on its SM and slow it.  MUON_PDL=2 turns it on for every call,
// MUON_PDL=0 off for every call.
void set_elementwise_pdl(bool on);
bool elementwise_pdl();

// Sets the option for the lifetime of the object, then restores it.
class ElementwisePdlScope {
 public:
  explicit ElementwisePdlScope(bool on) : old_(elementwise_pdl()) { set_elementwise_pdl(on); }
  ~ElementwisePdlScope() { set_elementwise_pdl(old_); }
  ElementwisePdlScope(const ElementwisePdlScope&) = delete;
  ElementwisePdlScope& operator=(const ElementwisePdlScope&) = delete;

 private:
  bool old_;
};

}  // namespace muon
