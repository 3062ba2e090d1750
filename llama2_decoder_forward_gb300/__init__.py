"""GB300 (sm_103a) Llama2 decoder forward: prefill and decode through a C ABI.

Submodules: `binding` (ctypes marshalling to libllama_gb300.so), `build`
(nvcc build of the library), `synth` (seeded synthetic inputs). Importing the
package loads nothing; `binding.lib()` loads the library on first use.
"""
