"""GB300 (sm_103a) fused multi-head latent attention.

The compute lives in the C-ABI library ``libmla_gb300.so`` (see include/mla.h);
``binding`` marshals torch tensors into it.  Import ``binding`` explicitly: it
raises if the library has not been built.
"""
__all__ = ["binding", "build"]
