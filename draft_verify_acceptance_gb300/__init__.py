"""GB300-native draft-then-verify acceptance step of speculative decoding.

The verify step runs in hand-written sm_103a CUDA kernels behind the C ABI
declared in ``include/spec_verify.h`` (library ``libspecverify.so``).  This
package holds that library's sources (``csrc/``), its build script, a thin
ctypes binding and the seeded input generators.

    from draft_verify_acceptance_gb300 import verify
    accepted_len, out_tokens = verify(target, draft, tokens, uniforms, 0.8, "sample")

Importing ``verify`` / ``verify_ex`` loads the library and raises ImportError
if it has not been built (``draft_verify_acceptance_gb300.build.build()``).
"""

__all__ = ["verify", "verify_ex", "workspace_size", "MODE_SAMPLE", "MODE_GREEDY"]

MODE_SAMPLE = 0
MODE_GREEDY = 1


def __getattr__(name):
    if name in ("verify", "verify_ex", "workspace_size", "binding"):
        import importlib
        binding = importlib.import_module(__name__ + ".binding")
        return binding if name == "binding" else getattr(binding, name)
    raise AttributeError(name)
